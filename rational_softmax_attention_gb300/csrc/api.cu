// The C ABI of libraattn (declared in include/raattn.h): argument validation,
// TMA tensor-map construction, the device status word, and dispatch to the
// kernels.  Nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "kernels.cuh"

namespace raattn {
namespace {

// One status word per device, read and cleared by ra_device_status().
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_force_timeout{0};
std::atomic<int> g_fwd_pair{0};
KernelEvents g_events = {{nullptr, nullptr, nullptr, nullptr}, 0};
std::mutex g_events_mu;

KernelEvents current_events() {
  std::lock_guard<std::mutex> lock(g_events_mu);
  return g_events;
}

ra_status_t status_ptr_for_current_device(unsigned int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return RA_ERR_LAUNCH;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status_ptr[dev];
  return RA_OK;
}

ra_status_t make_ctx(LaunchCtx* ctx) {
  unsigned int* p = nullptr;
  const ra_status_t st = status_ptr_for_current_device(&p);
  if (st != RA_OK) return st;
  ctx->status = p;
  ctx->wait_limit_ns = g_wait_limit_ns.load();
  ctx->force_timeout = g_force_timeout.load();
  return RA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Forward workspace: the fp16 copy of V, then (masked calls) the tile live map of up to B * H
// mask heads, 128-row query tiles by ceil(N_K / 128 / 32) words.  Each piece 256-byte padded.
int live_words_for(int NK) { return ((NK + 127) / 128 + 31) / 32; }
bool dtype_ok(ra_dtype_t t) { return t == RA_F32 || t == RA_BF16; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a [BH, N, D] 16-bit tensor: box {64, 128, 1}, 128-byte swizzle, zero fill
// out of bounds (rows past N of a head read as zeros, never the next head's rows).
bool make_map_16bit(CUtensorMap* map, const void* base, int BH, int N, int D, CUtensorMapDataType type,
                    cuuint32_t box_rows = 128) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(N) * D * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_map_bf16(CUtensorMap* map, const void* base, int BH, int N, int D) {
  return make_map_16bit(map, base, BH, N, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// Backward workspace.  CUDA-core path: D_i and R_i per row.  Tensor-core path: the
// per-query-tile constant blocks, then the fp16 copies of Q, dO, K and V.  Every piece
// starts on a 256-byte boundary.
struct BwdLayout {
  size_t per_row, consts, head, q16, kv16, live_q, live_k, plain_q, plain_k, total_f32, total_tc;
  BwdLayout(int B, int H, int NQ, int NK, int D) {
    auto pad = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    const size_t bh = static_cast<size_t>(B) * H;
    const size_t nqt = (static_cast<size_t>(NQ) + 127) / 128;
    per_row = pad(bh * NQ * sizeof(float));
    consts = pad(bh * nqt * kConstBlockFloats * sizeof(float));
    total_f32 = 2 * per_row;
    head = std::max(total_f32, consts);
    q16 = pad(bh * NQ * D * 2);
    kv16 = pad(bh * NK * D * 2);
    // masked calls: the tile live map by query tile (key-tile bits) and by key tile, then
    // the tile full map in the same two layouts, then one int per row of each layout
    const size_t nkt = (static_cast<size_t>(NK) + 127) / 128;
    live_q = pad(bh * nqt * live_words_for(NK) * 4);
    live_k = pad(bh * nkt * live_words_for(NQ) * 4);
    plain_q = pad(bh * nqt * 4);
    plain_k = pad(bh * nkt * 4);
    total_tc = head + 2 * q16 + 2 * kv16 + 2 * (live_q + live_k) + plain_q + plain_k;
  }
};

ra_status_t check_attn_sizes(int B, int H, int NQ, int NK, int D) {
  if (B < 1 || H < 1 || NQ < 1 || NK < 1 || D < 1) return RA_ERR_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > INT_MAX) return RA_ERR_ARG;
  // every per-tensor element index must fit comfortably in 64-bit arithmetic and
  // the per-head row counts in 32-bit
  if (bh * NQ > INT_MAX || bh * NK > INT_MAX) return RA_ERR_ARG;
  return RA_OK;
}

}  // namespace

size_t fwd_workspace_v_bytes(int B, int H, int NK, int D) {
  return (static_cast<size_t>(B) * H * NK * D * 2 + 255) & ~static_cast<size_t>(255);
}
size_t fwd_workspace_map_bytes(int B, int H, int NQ, int NK) {
  const size_t nqt = (static_cast<size_t>(NQ) + 127) / 128;
  return (static_cast<size_t>(B) * H * nqt * live_words_for(NK) * 4 + 255) & ~static_cast<size_t>(255);
}
size_t fwd_workspace_plain_bytes(int B, int H, int NQ) {
  const size_t nqt = (static_cast<size_t>(NQ) + 127) / 128;
  return (static_cast<size_t>(B) * H * nqt * 4 + 255) & ~static_cast<size_t>(255);
}
size_t fwd_workspace_live_bytes(int B, int H, int NQ, int NK) {
  return 2 * fwd_workspace_map_bytes(B, H, NQ, NK) + fwd_workspace_plain_bytes(B, H, NQ);
}

size_t bwd_workspace_bytes(int B, int H, int NQ, int NK, int D, bool f32_inputs) {
  if (check_attn_sizes(B, H, NQ, NK, D) != RA_OK) return 0;
  const BwdLayout lay(B, H, NQ, NK, D);
  return f32_inputs ? lay.total_f32 : lay.total_tc;
}

}  // namespace raattn

using namespace raattn;

extern "C" {

const char* ra_status_string(ra_status_t status) {
  switch (status) {
    case RA_OK: return "RA_OK";
    case RA_ERR_ARG: return "RA_ERR_ARG: invalid argument";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED: not implemented for these arguments";
    case RA_ERR_LAUNCH: return "RA_ERR_LAUNCH: CUDA launch or set-up failed";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT: a device-side wait exceeded its limit";
    default: return "unknown ra_status_t";
  }
}

void ra_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns == 0 ? 2000000000ull : static_cast<unsigned long long>(limit_ns));
}

void ra_debug_force_timeout(int on) { g_force_timeout.store(on ? 1 : 0); }

void ra_debug_fwd_pair(int mode) { g_fwd_pair.store(mode == 1 || mode == 2 ? mode : 0); }

void ra_debug_kernel_events(void* const* events, int n) {
  std::lock_guard<std::mutex> lock(g_events_mu);
  g_events.n = (events && n > 0) ? std::min(n, 4) : 0;
  for (int i = 0; i < 4; ++i) g_events.e[i] = i < g_events.n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
}

ra_status_t ra_device_status(void* stream) {
  unsigned int* p = nullptr;
  if (status_ptr_for_current_device(&p) != RA_OK) return RA_ERR_LAUNCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return RA_ERR_LAUNCH;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return RA_ERR_LAUNCH;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return RA_ERR_LAUNCH;
  if (v & kStatusBadSmem) return RA_ERR_LAUNCH;
  if (v & kStatusTimeout) return RA_ERR_TIMEOUT;
  return (v & kStatusRange) ? RA_ERR_UNSUPPORTED : RA_OK;
}

ra_status_t ra_softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols, ra_dtype_t dtype, void* stream) {
  if (!x || !y || rows < 1 || cols < 1 || !dtype_ok(dtype)) return RA_ERR_ARG;
  if (rows > INT_MAX || cols > (INT64_MAX / rows)) return RA_ERR_ARG;
  const cudaError_t e =
      dtype == RA_BF16
          ? launch_ra_softmax_fwd_bf16(x, y, rows, cols, static_cast<cudaStream_t>(stream))
          : launch_ra_softmax_fwd_f32(static_cast<const float*>(x), static_cast<float*>(y), rows, cols,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

ra_status_t ra_softmax_bwd(const void* x, const void* p, const void* dy, void* dx, int64_t rows, int64_t cols,
                           ra_dtype_t dtype, void* stream) {
  if (!x || !p || !dy || !dx || rows < 1 || cols < 1 || !dtype_ok(dtype)) return RA_ERR_ARG;
  if (rows > INT_MAX || cols > (INT64_MAX / rows)) return RA_ERR_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dtype == RA_F32 ? launch_ra_softmax_bwd_f32(static_cast<const float*>(x), static_cast<const float*>(p),
                                                  static_cast<const float*>(dy), static_cast<float*>(dx), rows, cols,
                                                  st)
                      : launch_ra_softmax_bwd_bf16(x, p, dy, dx, rows, cols, st);
  return e == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

size_t ra_attention_fwd_workspace_size(int B, int H, int N_Q, int N_K, int D) {
  if (check_attn_sizes(B, H, N_Q, N_K, D) != RA_OK) return 0;
  return raattn::fwd_workspace_v_bytes(B, H, N_K, D) + raattn::fwd_workspace_live_bytes(B, H, N_Q, N_K);
}

}  // extern "C"

namespace raattn {
namespace {

// Validates a packed mask for (B, H, N_Q, N_K); fills `m` (bits null when there is no mask).
ra_status_t mask_args(const uint32_t* bits, int MB, int MH, int B, int H, int cols, MaskBits* m) {
  m->bits = bits;
  m->words = ra_attention_mask_words(cols);
  m->mb = MB;
  m->mh = MH;
  m->live = nullptr;
  m->full = nullptr;
  m->plain = nullptr;
  m->live_words = 0;
  if (!bits) return RA_OK;
  if (!aligned16(bits) || !(MB == 1 || MB == B) || !(MH == 1 || MH == H)) return RA_ERR_ARG;
  return RA_OK;
}

ra_status_t attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* row_m, float* row_s,
                          int32_t* row_arg, int64_t* tile_counts, void* workspace, int B, int H, int N_Q, int N_K,
                          int D, float scale, int causal, ra_dtype_t in_dtype, ra_dtype_t out_dtype, void* stream,
                          const MaskBits& mask) {
  if (!q || !k || !v || !o || !dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return RA_ERR_ARG;
  if (check_attn_sizes(B, H, N_Q, N_K, D) != RA_OK) return RA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return RA_ERR_ARG;
  if ((row_m && !aligned16(row_m)) || (row_s && !aligned16(row_s)) || (row_arg && !aligned16(row_arg)) ||
      (tile_counts && !aligned16(tile_counts)) || (workspace && !aligned16(workspace)))
    return RA_ERR_ARG;
  if (in_dtype == RA_BF16 && !workspace) return RA_ERR_ARG;   // the tensor-core path needs the fp16 V copy
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(scale)) return RA_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AttnShape s{B, H, N_Q, N_K, D, scale, causal ? 1 : 0};

  if (in_dtype == RA_F32) {
    if (!(D == 16 || D == 32 || D == 64 || D == 128)) return RA_ERR_UNSUPPORTED;
    if (mask.bits) return RA_ERR_UNSUPPORTED;   // masks on the tensor-core (bf16) path only
    if (tile_counts && cudaMemsetAsync(tile_counts, 0, 2 * sizeof(int64_t), st) != cudaSuccess) return RA_ERR_LAUNCH;
    const cudaError_t e = launch_attn_fwd_simt(s, static_cast<const float*>(q), static_cast<const float*>(k),
                                               static_cast<const float*>(v), o, out_dtype == RA_BF16, row_m, row_s,
                                               row_arg, st);
    return e == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
  }
  // bf16: tensor-core path
  if (!(D == 64 || D == 128)) return RA_ERR_UNSUPPORTED;
  LaunchCtx ctx;
  if (make_ctx(&ctx) != RA_OK) return RA_ERR_LAUNCH;
  FwdTcArgs a;
  const int BH = B * H;
  if (!make_map_bf16(&a.tm_q, q, BH, N_Q, D) || !make_map_bf16(&a.tm_k, k, BH, N_K, D) ||
      !make_map_16bit(&a.tm_k64, k, BH, N_K, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64) ||
      !make_map_16bit(&a.tm_v, workspace, BH, N_K, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
    return RA_ERR_LAUNCH;
  const int pair_mode = g_fwd_pair.load();
  a.pair = D == 128 && (pair_mode == 2 || (pair_mode == 0 && N_Q > 256)) ? 1 : 0;
  ConvertJob job;
  job.src[0] = static_cast<const uint4*>(v);
  job.dst[0] = static_cast<uint4*>(workspace);
  job.n8[0] = static_cast<size_t>(BH) * N_K * D / 8;
  job.count = 1;
  a.o = o;
  a.row_m = row_m;
  a.row_s = row_s;
  a.row_arg = row_arg;
  a.tile_counts = reinterpret_cast<unsigned long long*>(tile_counts);
  a.out_bf16 = out_dtype == RA_BF16 ? 1 : 0;
  a.mask = mask;
  if (mask.bits) {   // tile maps after the V copy: fully masked tiles are left out of both passes,
                     // wholly allowed ones read no mask words
    char* maps = static_cast<char*>(workspace) + fwd_workspace_v_bytes(B, H, N_K, D);
    const size_t map_bytes = fwd_workspace_map_bytes(B, H, N_Q, N_K);
    uint32_t* live = reinterpret_cast<uint32_t*>(maps);
    uint32_t* full = reinterpret_cast<uint32_t*>(maps + map_bytes);
    int* plain = reinterpret_cast<int*>(maps + 2 * map_bytes);
    a.mask.live = live;
    a.mask.full = full;
    a.mask.plain = plain;
    a.mask.live_words = live_words_for(N_K);
    if (launch_mask_tile_live(mask.bits, mask.mb * mask.mh, N_Q, N_K, mask.words, causal ? 1 : 0, live, full, plain,
                              a.mask.live_words, nullptr, nullptr, nullptr, 0, st) != cudaSuccess)
      return RA_ERR_LAUNCH;
  }
  if (tile_counts && cudaMemsetAsync(tile_counts, 0, 2 * sizeof(int64_t), st) != cudaSuccess) return RA_ERR_LAUNCH;
  const KernelEvents ev = current_events();
  if (ev.rec(0, st) != cudaSuccess) return RA_ERR_LAUNCH;
  if (launch_bf16_to_f16(job, ctx.status, st) != cudaSuccess) return RA_ERR_LAUNCH;
  if (ev.rec(1, st) != cudaSuccess) return RA_ERR_LAUNCH;
  const cudaError_t e = launch_attn_fwd_tc(s, a, ctx, st);
  if (e != cudaSuccess || ev.rec(2, st) != cudaSuccess) return RA_ERR_LAUNCH;
  return RA_OK;
}

}  // namespace
}  // namespace raattn

extern "C" {

ra_status_t ra_attention_fwd(const void* q, const void* k, const void* v, void* o, float* row_m, float* row_s,
                             int32_t* row_arg, int64_t* tile_counts, void* workspace, int B, int H, int N_Q,
                             int N_K, int D, float scale, int causal, ra_dtype_t in_dtype, ra_dtype_t out_dtype,
                             void* stream) {
  const MaskBits none{nullptr, 0, 1, 1, nullptr, nullptr, nullptr, 0};
  return attn_fwd_impl(q, k, v, o, row_m, row_s, row_arg, tile_counts, workspace, B, H, N_Q, N_K, D, scale, causal,
                       in_dtype, out_dtype, stream, none);
}

ra_status_t ra_attention_fwd_masked(const void* q, const void* k, const void* v, void* o, float* row_m,
                                    float* row_s, int32_t* row_arg, int64_t* tile_counts, void* workspace, int B,
                                    int H, int N_Q, int N_K, int D, float scale, int causal, ra_dtype_t in_dtype,
                                    ra_dtype_t out_dtype, const uint32_t* mask_q, int MB, int MH, void* stream) {
  if (!mask_q) return RA_ERR_ARG;
  MaskBits m;
  const ra_status_t r = mask_args(mask_q, MB, MH, B, H, N_K, &m);
  if (r != RA_OK) return r;
  return attn_fwd_impl(q, k, v, o, row_m, row_s, row_arg, tile_counts, workspace, B, H, N_Q, N_K, D, scale, causal,
                       in_dtype, out_dtype, stream, m);
}

int ra_attention_mask_words(int n) { return n < 1 ? 0 : ((n + 127) / 128) * 4; }

ra_status_t ra_attention_mask_pack(const void* mask, int G, int N_Q, int N_K, uint32_t* bits_q, uint32_t* bits_k,
                                   void* stream) {
  if (!mask || (!bits_q && !bits_k) || G < 1 || N_Q < 1 || N_K < 1) return RA_ERR_ARG;
  if (static_cast<long long>(G) * N_Q * N_K > (1ll << 40)) return RA_ERR_ARG;
  if ((bits_q && !aligned16(bits_q)) || (bits_k && !aligned16(bits_k))) return RA_ERR_ARG;
  const cudaError_t e = launch_mask_pack(static_cast<const uint8_t*>(mask), G, N_Q, N_K, bits_q,
                                         ra_attention_mask_words(N_K), bits_k, ra_attention_mask_words(N_Q),
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

size_t ra_attention_bwd_workspace_size(int B, int H, int N_Q, int N_K, int D) {
  if (check_attn_sizes(B, H, N_Q, N_K, D) != RA_OK) return 0;
  return BwdLayout(B, H, N_Q, N_K, D).total_tc;   // enough for either path
}

}  // extern "C"

namespace raattn {
namespace {

ra_status_t attn_bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* row_m, const float* row_s, const int32_t* row_arg, void* dq, void* dk,
                          void* dv, void* workspace, int B, int H, int N_Q, int N_K, int D, float scale, int causal,
                          ra_dtype_t in_dtype, ra_dtype_t o_dtype, ra_dtype_t grad_dtype, void* stream,
                          const MaskBits& mask_q, const MaskBits& mask_k) {
  if (!q || !k || !v || !o || !dout || !row_m || !row_s || !row_arg || !dq || !dk || !dv || !workspace)
    return RA_ERR_ARG;
  if (!dtype_ok(in_dtype) || !dtype_ok(o_dtype) || !dtype_ok(grad_dtype)) return RA_ERR_ARG;
  if (check_attn_sizes(B, H, N_Q, N_K, D) != RA_OK) return RA_ERR_ARG;
  const void* ptrs[] = {q, k, v, o, dout, row_m, row_s, row_arg, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return RA_ERR_ARG;
  if (!(scale > 0.0f)) scale = 1.0f / std::sqrt(static_cast<float>(D));
  if (!std::isfinite(scale)) return RA_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AttnShape s{B, H, N_Q, N_K, D, scale, causal ? 1 : 0};
  const BwdLayout lay(B, H, N_Q, N_K, D);
  const size_t per = lay.per_row;
  char* ws = static_cast<char*>(workspace);
  float* ws_d = reinterpret_cast<float*>(ws);
  float* ws_r = reinterpret_cast<float*>(ws + per);

  if (in_dtype == RA_F32) {
    if (!(D == 16 || D == 32 || D == 64 || D == 128)) return RA_ERR_UNSUPPORTED;
    if (mask_q.bits) return RA_ERR_UNSUPPORTED;   // masks on the tensor-core (bf16) path only
    const cudaError_t e = launch_attn_bwd_simt(
        s, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), o,
        o_dtype == RA_BF16, static_cast<const float*>(dout), row_m, row_s, row_arg, dq, dk, dv,
        grad_dtype == RA_BF16, ws_d, ws_r, st);
    return e == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
  }
  if (!(D == 64 || D == 128)) return RA_ERR_UNSUPPORTED;
  LaunchCtx ctx;
  if (make_ctx(&ctx) != RA_OK) return RA_ERR_LAUNCH;
  BwdTcArgs a;
  const int BH = B * H;
  a.q16 = ws + lay.head;
  a.do16 = ws + lay.head + lay.q16;
  a.k16 = ws + lay.head + 2 * lay.q16;
  a.v16 = ws + lay.head + 2 * lay.q16 + lay.kv16;
  const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!make_map_16bit(&a.tm_q, a.q16, BH, N_Q, D, f16) || !make_map_16bit(&a.tm_k, a.k16, BH, N_K, D, f16) ||
      !make_map_16bit(&a.tm_v, a.v16, BH, N_K, D, f16) || !make_map_16bit(&a.tm_do, a.do16, BH, N_Q, D, f16))
    return RA_ERR_LAUNCH;
  a.v_raw = v;
  a.o = o;
  a.o_bf16 = o_dtype == RA_BF16 ? 1 : 0;
  a.dout = dout;
  a.row_m = row_m;
  a.row_s = row_s;
  a.row_arg = row_arg;
  a.k_raw = k;
  a.q_raw = q;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.grad_bf16 = grad_dtype == RA_BF16 ? 1 : 0;
  a.ws_consts = reinterpret_cast<float*>(ws);
  a.mask_q = mask_q;
  a.mask_k = mask_k;
  if (mask_q.bits) {   // the tile maps, both ways: fully masked tiles are left out of both kernels,
                       // wholly allowed ones read no mask words
    char* lq = ws + lay.head + 2 * lay.q16 + 2 * lay.kv16;
    uint32_t* live_q = reinterpret_cast<uint32_t*>(lq);
    uint32_t* live_k = reinterpret_cast<uint32_t*>(lq + lay.live_q);
    uint32_t* full_q = reinterpret_cast<uint32_t*>(lq + lay.live_q + lay.live_k);
    uint32_t* full_k = reinterpret_cast<uint32_t*>(lq + 2 * lay.live_q + lay.live_k);
    int* plain_q = reinterpret_cast<int*>(lq + 2 * (lay.live_q + lay.live_k));
    int* plain_k = reinterpret_cast<int*>(lq + 2 * (lay.live_q + lay.live_k) + lay.plain_q);
    a.mask_q.live = live_q;
    a.mask_q.full = full_q;
    a.mask_q.plain = plain_q;
    a.mask_q.live_words = live_words_for(N_K);
    a.mask_k.live = live_k;
    a.mask_k.full = full_k;
    a.mask_k.plain = plain_k;
    a.mask_k.live_words = live_words_for(N_Q);
    if (launch_mask_tile_live(mask_q.bits, mask_q.mb * mask_q.mh, N_Q, N_K, mask_q.words, causal ? 1 : 0, live_q,
                              full_q, plain_q, a.mask_q.live_words, live_k, full_k, plain_k, a.mask_k.live_words,
                              st) != cudaSuccess)
      return RA_ERR_LAUNCH;
  }
  const cudaError_t e = launch_attn_bwd_tc(s, a, ctx, st, current_events());
  return e == cudaSuccess ? RA_OK : RA_ERR_LAUNCH;
}

}  // namespace
}  // namespace raattn

extern "C" {

ra_status_t ra_attention_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                             const float* row_m, const float* row_s, const int32_t* row_arg, void* dq, void* dk,
                             void* dv, void* workspace, int B, int H, int N_Q, int N_K, int D, float scale,
                             int causal, ra_dtype_t in_dtype, ra_dtype_t o_dtype, ra_dtype_t grad_dtype,
                             void* stream) {
  const MaskBits none{nullptr, 0, 1, 1, nullptr, nullptr, nullptr, 0};
  return attn_bwd_impl(q, k, v, o, dout, row_m, row_s, row_arg, dq, dk, dv, workspace, B, H, N_Q, N_K, D, scale,
                       causal, in_dtype, o_dtype, grad_dtype, stream, none, none);
}

ra_status_t ra_attention_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                    const float* row_m, const float* row_s, const int32_t* row_arg, void* dq,
                                    void* dk, void* dv, void* workspace, int B, int H, int N_Q, int N_K, int D,
                                    float scale, int causal, ra_dtype_t in_dtype, ra_dtype_t o_dtype,
                                    ra_dtype_t grad_dtype, const uint32_t* mask_q, const uint32_t* mask_k, int MB,
                                    int MH, void* stream) {
  if (!mask_q || !mask_k) return RA_ERR_ARG;
  MaskBits mq, mk;
  ra_status_t r = mask_args(mask_q, MB, MH, B, H, N_K, &mq);
  if (r == RA_OK) r = mask_args(mask_k, MB, MH, B, H, N_Q, &mk);
  if (r != RA_OK) return r;
  return attn_bwd_impl(q, k, v, o, dout, row_m, row_s, row_arg, dq, dk, dv, workspace, B, H, N_Q, N_K, D, scale,
                       causal, in_dtype, o_dtype, grad_dtype, stream, mq, mk);
}

}  // extern "C"
