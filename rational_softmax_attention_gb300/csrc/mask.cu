// Bit-packing of a boolean attention mask for the tensor-core attention kernels.
//
// Page "Ra-Family: Rational Neural Architecture", section 3, ra_attention: a drop-in for
// scaled_dot_product_attention, whose boolean attn_mask marks with True the (query, key)
// pairs that take part.  The kernels read the mask one 32-column word per row and tile
// chunk: bits_q with a row per query (forward, dQ kernel) and bits_k with a row per key
// (dK/dV kernel, whose threads own key rows).  A tile live map (one bit per 128 x 128 block
// with any allowed pair) lets a kernel leave fully masked tiles out altogether, and a tile
// full map (every pair below N_Q and N_K allowed) lets it treat such a block as unmasked,
// reading no mask words.
#include "kernels.cuh"

namespace raattn {
namespace {

constexpr int WARPS = 8;

// One warp per (mask head, query row, word): lane l reads column 32 w + l, the ballot is the word.
__global__ void __launch_bounds__(32 * WARPS) mask_pack_rows_kernel(const uint8_t* mask, int NQ, int NK,
                                                                    uint32_t* bits, int words, long long total) {
  const long long wid = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= total) return;   // uniform across the warp
  const int w = static_cast<int>(wid % words);
  const long long row = wid / words;   // g * NQ + i
  const int c = 32 * w + lane;
  const bool on = c < NK && mask[row * NK + c] != 0;
  const uint32_t word = __ballot_sync(0xffffffffu, on);
  if (lane == 0) bits[row * words + w] = word;
}

// One warp per (mask head, query word w, block of 32 keys): lane l builds the word of key
// j0 + l from rows 32 w .. 32 w + 31, reading 32 consecutive bytes of each row.
__global__ void __launch_bounds__(32 * WARPS) mask_pack_cols_kernel(const uint8_t* mask, int NQ, int NK,
                                                                    uint32_t* bits, int words, int kblocks,
                                                                    long long total) {
  const long long wid = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= total) return;
  const int kb = static_cast<int>(wid % kblocks);
  const long long rest = wid / kblocks;
  const int w = static_cast<int>(rest % words);
  const long long g = rest / words;
  const int j = 32 * kb + lane;
  uint32_t word = 0;
  for (int r = 0; r < 32; ++r) {
    const int i = 32 * w + r;
    if (i < NQ && j < NK && mask[(g * NQ + i) * NK + j] != 0) word |= 1u << r;
  }
  if (j < NK) bits[(g * NK + j) * words + w] = word;
}

// One warp per (mask head, query tile, key tile): the block is live when any of the query
// tile's rows may attend to any key of the tile, and full when every row may attend to every
// key of it below N_K, read from the packed rows (four words per key tile).  Lane l scans
// rows l, l + 32, l + 64, l + 96 of the query tile (those below N_Q).  A live block sets bit
// kt of its query tile's row of live_q (key tiles along the row) and, when live_k is given,
// bit qt of its key tile's row of live_k (the same map transposed); a full one the same bits
// of full_q and full_k.  The kernels check N_K and N_Q themselves, so a full block past
// either edge is treated as unmasked there.
__global__ void __launch_bounds__(32 * WARPS) mask_tile_live_kernel(const uint32_t* bits_q, int NQ, int NK,
                                                                    int words, int nqt, int nkt, uint32_t* live_q,
                                                                    uint32_t* full_q, int wq, uint32_t* live_k,
                                                                    uint32_t* full_k, int wk, long long total) {
  const long long wid = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= total) return;   // uniform across the warp
  const int kt = static_cast<int>(wid % nkt);
  const long long rest = wid / nkt;   // g * nqt + qt
  const int qt = static_cast<int>(rest % nqt);
  const long long g = rest / nqt;
  // bits of the columns past N_K, which count as allowed for the full test
  uint32_t pad[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int c0 = kt * 128 + 32 * w;   // first column of word w
    const int n_in = min(max(NK - c0, 0), 32);
    pad[w] = n_in >= 32 ? 0u : ~((1u << n_in) - 1u);
  }
  uint32_t any = 0, all = ~0u;
  for (int r = lane; r < 128; r += 32) {
    const int i = qt * 128 + r;
    if (i < NQ) {
      const uint4 u = *reinterpret_cast<const uint4*>(bits_q + (g * NQ + i) * words + 4 * kt);
      any |= u.x | u.y | u.z | u.w;
      all &= (u.x | pad[0]) & (u.y | pad[1]) & (u.z | pad[2]) & (u.w | pad[3]);
    }
  }
  const bool on = __any_sync(0xffffffffu, any != 0);
  const bool whole = __all_sync(0xffffffffu, all == ~0u);   // row qt * 128 < N_Q: whole implies on
  if (lane == 0 && on) {
    atomicOr(&live_q[rest * wq + kt / 32], 1u << (kt % 32));
    if (live_k) atomicOr(&live_k[(g * nkt + kt) * wk + qt / 32], 1u << (qt % 32));
  }
  if (lane == 0 && whole) {
    if (full_q) atomicOr(&full_q[rest * wq + kt / 32], 1u << (kt % 32));
    if (full_k) atomicOr(&full_k[(g * nkt + kt) * wk + qt / 32], 1u << (qt % 32));
  }
}

// One thread per row of the tile maps.  Rows of query tiles: plain_q = n when the live row
// equals the full row and is key tiles 0 .. n - 1 (a key-padding mask, or an all-true one:
// every row of the query tile may see exactly the keys before 128 n, so an unmasked kernel
// over those keys gives the masked results), else 0.  Rows of key tiles: plain_k = 1 when the
// full row holds every query tile from qt0 = (causal ? kt : 0) on, the query tiles a key tile
// of the unmasked kernels takes, else 0.
__global__ void __launch_bounds__(256) mask_tile_plain_kernel(const uint32_t* live_q, const uint32_t* full_q, int wq,
                                                              int nqt, int* plain_q, const uint32_t* full_k, int wk,
                                                              int nkt, int* plain_k, int causal, long long rows_q,
                                                              long long total) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= total) return;
  if (t < rows_q) {
    const uint32_t* L = live_q + t * wq;
    const uint32_t* F = full_q + t * wq;
    int n = 0;
    bool ok = true, ended = false;   // ended: a clear bit seen, every later bit must be clear
    for (int w = 0; w < wq && ok; ++w) {
      const uint32_t l = L[w];
      ok = l == F[w] && (ended ? l == 0u : (l & (l + 1u)) == 0u);   // 0..01..1 before the end
      if (!ended) n += __popc(l);
      ended = ended || l != ~0u;
    }
    plain_q[t] = ok ? n : 0;
  } else {
    const long long r = t - rows_q;   // g * nkt + kt
    const int kt = static_cast<int>(r % nkt);
    const int qt0 = causal ? kt : 0;   // 128-row query tiles and 128-key tiles
    const uint32_t* F = full_k + r * wk;
    bool ok = true;
    for (int w = 0; w < wk && ok; ++w) {
      const int lo = min(max(qt0 - 32 * w, 0), 32), hi = min(max(nqt - 32 * w, 0), 32);
      const uint32_t upto_hi = hi >= 32 ? ~0u : (1u << hi) - 1u;
      const uint32_t from_lo = lo >= 32 ? 0u : ~((1u << lo) - 1u);
      const uint32_t range = upto_hi & from_lo;
      ok = (F[w] & range) == range;
    }
    plain_k[r] = ok ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_mask_tile_live(const uint32_t* bits_q, int G, int NQ, int NK, int words, int causal,
                                  uint32_t* live_q, uint32_t* full_q, int* plain_q, int wq, uint32_t* live_k,
                                  uint32_t* full_k, int* plain_k, int wk, cudaStream_t st) {
  const int nqt = (NQ + 127) / 128, nkt = (NK + 127) / 128;
  const size_t bytes_q = static_cast<size_t>(G) * nqt * wq * sizeof(uint32_t);
  const size_t bytes_k = static_cast<size_t>(G) * nkt * wk * sizeof(uint32_t);
  cudaError_t e = cudaMemsetAsync(live_q, 0, bytes_q, st);
  if (e == cudaSuccess && full_q) e = cudaMemsetAsync(full_q, 0, bytes_q, st);
  if (e == cudaSuccess && live_k) e = cudaMemsetAsync(live_k, 0, bytes_k, st);
  if (e == cudaSuccess && full_k) e = cudaMemsetAsync(full_k, 0, bytes_k, st);
  if (e != cudaSuccess) return e;
  const long long total = static_cast<long long>(G) * nqt * nkt;
  const unsigned grid = static_cast<unsigned>((total + WARPS - 1) / WARPS);
  mask_tile_live_kernel<<<grid, 32 * WARPS, 0, st>>>(bits_q, NQ, NK, words, nqt, nkt, live_q, full_q, wq, live_k,
                                                     full_k, wk, total);
  e = cudaGetLastError();
  if (e != cudaSuccess || !plain_q || !full_q) return e;
  const long long rows_q = static_cast<long long>(G) * nqt;
  const long long rows = rows_q + (plain_k && full_k ? static_cast<long long>(G) * nkt : 0);
  mask_tile_plain_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(
      live_q, full_q, wq, nqt, plain_q, full_k, wk, nkt, plain_k, causal, rows_q, rows);
  return cudaGetLastError();
}

cudaError_t launch_mask_pack(const uint8_t* mask, int G, int NQ, int NK, uint32_t* bits_q, int wq, uint32_t* bits_k,
                             int wk, cudaStream_t st) {
  if (bits_q) {
    const long long total = static_cast<long long>(G) * NQ * wq;
    const unsigned grid = static_cast<unsigned>((total + WARPS - 1) / WARPS);
    mask_pack_rows_kernel<<<grid, 32 * WARPS, 0, st>>>(mask, NQ, NK, bits_q, wq, total);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (bits_k) {
    const int kblocks = (NK + 31) / 32;
    const long long total = static_cast<long long>(G) * wk * kblocks;
    const unsigned grid = static_cast<unsigned>((total + WARPS - 1) / WARPS);
    mask_pack_cols_kernel<<<grid, 32 * WARPS, 0, st>>>(mask, NQ, NK, bits_k, wk, kblocks, total);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace raattn
