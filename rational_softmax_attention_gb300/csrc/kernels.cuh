// Launchers exported by each kernel translation unit to the C-ABI layer (api.cu).
#pragma once

#include <cuda.h>
#include "common.cuh"

namespace raattn {

// ra_softmax (ra_softmax.cu)
cudaError_t launch_ra_softmax_fwd_f32(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t st);
cudaError_t launch_ra_softmax_fwd_bf16(const void* x, void* y, int64_t rows, int64_t cols, cudaStream_t st);
cudaError_t launch_ra_softmax_bwd_f32(const float* x, const float* p, const float* dy, float* dx, int64_t rows,
                                      int64_t cols, cudaStream_t st);
cudaError_t launch_ra_softmax_bwd_bf16(const void* x, const void* p, const void* dy, void* dx, int64_t rows,
                                       int64_t cols, cudaStream_t st);

// Boolean attention mask, bit-packed: bit (c % 32) of word c / 32 of a row is set when that
// column may be attended.  Rows of `words` uint32 (a multiple of 4: whole 128-column tiles,
// 16-byte aligned), one [rows x words] matrix per mask head g = (mb > 1 ? b : 0) * mh +
// (mh > 1 ? h : 0), so a mask can be shared across the batch and/or the heads.
struct MaskBits {
  const uint32_t* bits;   // null: no mask
  int words;
  int mb, mh;
  const uint32_t* live;   // optional tile live map of the same mask heads (null: every tile may be live)
  const uint32_t* full;   // optional map of the tiles whose every pair is allowed, laid out like `live`
  const int* plain;       // optional, one per row of the maps: a row an unmasked call can serve (mask.cu)
  int live_words;         // words per query tile row of the maps
};
// Packs a [G, NQ, NK] byte mask (nonzero = may attend) into bits_q [G, NQ, wq] (rows = queries)
// and bits_k [G, NK, wk] (rows = keys); either may be null (mask.cu).
cudaError_t launch_mask_pack(const uint8_t* mask, int G, int NQ, int NK, uint32_t* bits_q, int wq, uint32_t* bits_k,
                             int wk, cudaStream_t st);
// Tile maps from packed query rows (bits_q, `words` per row): for mask head g, bit kt of
// live_q[(g * nqt + qt) * wq + kt / 32] is set when any pair of the 128 x 128 block (query tile
// qt, key tile kt) may attend, and the same bit of full_q when every pair of it below N_Q
// and N_K may;
// live_k and full_k (optional) hold the transposes, bit qt of [(g * nkt + kt) * wk + qt / 32].
// Then, per row, plain_q[g * nqt + qt] = n > 0 when query tile qt's live and full rows are
// both key tiles 0 .. n - 1 (else 0), and (with the transposes) plain_k[g * nkt + kt] = 1 when
// every query tile of key tile kt's range (from kt on when causal, else all) is full (mask.cu).
cudaError_t launch_mask_tile_live(const uint32_t* bits_q, int G, int NQ, int NK, int words, int causal,
                                  uint32_t* live_q, uint32_t* full_q, int* plain_q, int wq, uint32_t* live_k,
                                  uint32_t* full_k, int* plain_k, int wk, cudaStream_t st);

// Caller-supplied CUDA events recorded at an attention call's kernel boundaries (a
// measurement knob, ra_debug_kernel_events): e[i] is recorded before kernel i of the call
// and e[k] after its last kernel k - 1; null entries and i >= n are skipped.
struct KernelEvents {
  cudaEvent_t e[4];
  int n;
  cudaError_t rec(int i, cudaStream_t st) const {
    return (i < n && e[i]) ? cudaEventRecord(e[i], st) : cudaSuccess;
  }
};

// Problem description shared by the attention launchers.
struct AttnShape {
  int B, H, NQ, NK, D;
  float scale;   // > 0 (the C-ABI layer resolves the default)
  int causal;
};

// fp32 CUDA-core attention (attn_simt.cu).  out_bf16 selects the output dtype.
cudaError_t launch_attn_fwd_simt(const AttnShape& s, const float* q, const float* k, const float* v, void* o,
                                 bool out_bf16, float* row_m, float* row_s, int32_t* row_arg, cudaStream_t st);
cudaError_t launch_attn_bwd_simt(const AttnShape& s, const float* q, const float* k, const float* v,
                                 const void* o, bool o_bf16, const float* dout, const float* row_m,
                                 const float* row_s, const int32_t* row_arg, void* dq, void* dk, void* dv,
                                 bool grad_bf16, float* ws_d, float* ws_r, cudaStream_t st);

// bf16 -> fp16 copies of up to four tensors in one launch (convert.cu).  n8 = elements / 8.
struct ConvertJob {
  const uint4* src[4];
  uint4* dst[4];
  size_t n8[4];
  int count;
};
cudaError_t launch_bf16_to_f16(const ConvertJob& job, unsigned int* status, cudaStream_t st);

// bf16 tensor-core attention forward (attn_fwd_tc.cu).  Tensor maps are built by the caller.
struct FwdTcArgs {
  CUtensorMap tm_q, tm_k;   // bf16 Q and K: 3-D maps {D, N, B*H}, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tm_v;         // fp16 copy of V (same geometry)
  CUtensorMap tm_k64;       // K with 64-row boxes {64, 64, 1} (CTA pair form)
  void* o;
  float* row_m;
  float* row_s;
  int32_t* row_arg;
  unsigned long long* tile_counts;   // may be null
  int out_bf16;
  MaskBits mask;   // rows = queries
  int pair;        // D = 128: run as CTA pairs (cta_group::2 products)
};
cudaError_t launch_attn_fwd_tc(const AttnShape& s, const FwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st);

// bf16 tensor-core attention backward (attn_bwd_tc.cu).
struct BwdTcArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;   // same geometry as the forward maps
  const void* o;
  int o_bf16;
  const void* dout;
  const float* row_m;
  const float* row_s;
  const int32_t* row_arg;
  const void* k_raw;   // K in global memory (bf16), for the argmax correction
  const void* q_raw;   // Q in global memory (bf16)
  const void* v_raw;   // V in global memory (bf16)
  void* q16;           // fp16 copies in the workspace, read through the tensor maps
  void* k16;
  void* v16;
  void* do16;
  void* dq;
  void* dk;
  void* dv;
  int grad_bf16;
  // Per-query constants, one 2560-byte block per (batch*head, 128-row query tile), written
  // by the dQ kernel and bulk-copied by the dK/dV kernel: [5][128] of
  //   base_i = 0.5 + scale * row_m_i / 32 (so w = (1+u)/2 = base_i - scale * s / 32),
  //   1 / row_s_i, D_i / 4 (D_i = dO_i . O_i), R_i = sum_j E_ij (argmax excluded), and
  //   the argmax index a_i (int32 bits); rows past N_Q hold 2, 0, 0, 0, -1.
  float* ws_consts;
  MaskBits mask_q;   // rows = queries (dQ kernel)
  MaskBits mask_k;   // the same mask transposed, rows = keys (dK/dV kernel)
};
constexpr int kConstBlockFloats = 5 * 128;
// Forward workspace pieces (api.cu): the fp16 copy of V, and the tile maps of a masked call
// (the live map, then the full map, each fwd_workspace_map_bytes, then the per-row plain
// lengths, fwd_workspace_plain_bytes).
size_t fwd_workspace_v_bytes(int B, int H, int NK, int D);
size_t fwd_workspace_map_bytes(int B, int H, int NQ, int NK);
size_t fwd_workspace_plain_bytes(int B, int H, int NQ);
size_t fwd_workspace_live_bytes(int B, int H, int NQ, int NK);
// Workspace bytes the backward uses for these sizes and input dtype (api.cu): the CUDA-core
// fp32 path needs only two per-row float arrays; the tensor-core path the constant blocks and
// the fp16 operand copies.  0 for invalid sizes.
size_t bwd_workspace_bytes(int B, int H, int NQ, int NK, int D, bool f32_inputs);
// Kernels in launch order: bf16 -> fp16 operand copies, dQ kernel, dK/dV kernel.
cudaError_t launch_attn_bwd_tc(const AttnShape& s, const BwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st,
                               const KernelEvents& ev);

}  // namespace raattn
