// bf16 ra_attention forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Page "Ra-Family: Rational Neural Architecture", section 3, ra_attention:
// (Q, K, V) -> O without storing [B, H, N_Q, N_K]; a two-pass tiled kernel that
// skips the V tile and its product whenever every entry of a tile lies outside
// the compact support (min u >= 1).  Section 3, ra_softmax: phi = ((1-u)/(1+u))^8
// for u < 1, exactly 0 otherwise, u = (x_max - x)/16.
//
// Why two passes: phi(Delta + c) is not phi(Delta) times a function of c, so the
// running-max rescaling of standard flash attention does not exist here; the
// row maximum must be final before any phi is formed.
//
// One CTA owns one 128-row query tile of one (batch, head) and runs both passes
// over the key tiles that the tile can see (all of them, or up to the diagonal
// when causal), so Q stays in shared memory and m_i stays in a register:
//   warp 4      TMA producer: Q once, then K tiles (pass 1), then K and V tiles
//               interleaved in the order the MMA warp consumes them (pass 2),
//               through a ring of NSTAGE shared-memory stages.
//   warp 5      MMA issuer (one thread): S = Q K^T into one of two TMEM score
//               buffers (128 x 128 fp32), and in pass 2 O += P V into a TMEM
//               accumulator (128 x D fp32), one K step behind the scores so the
//               tensor core computes S_{j+1} while the softmax warps work on S_j.
//   warps 0-3   softmax warpgroup, thread t owns query row t (TMEM lane t):
//               pass 1 reads S and keeps the running max and lowest argmax;
//               pass 2 reads S, forms phi on the FMA pipe (no exp), writes
//               P = fp16(phi) into a 128-byte-swizzled shared-memory tile for the
//               P V product, sums phi in fp32, and votes whether the tile is live.
//               Epilogue: O = acc / sum(phi), row statistics for the backward.
//   V arrives as the fp16 copy the C-ABI layer made once per call (exact for bf16
//   values up to 65504), so the P V product runs in fp16 and P is rounded to 2^-11
//   rather than 2^-8.  Q K^T stays in bf16.
//
// phi on the FMA pipe: w = (1+u)/2 = 0.5 + (m - s)/32 (scaled units) computed with
// one saturating FMA, so every u >= 1 (and every masked entry, fed as -inf) gives
// w = 1; q = 1/w - 1; phi = ((q^2)^2)^2.  The reciprocals are taken two at a
// time from one rcp.approx of w0*w1 (then 1/w0 = R w1, 1/w1 = R w0), halving the
// special-function-unit work, and the rest runs as packed f32x2 operations.
// At w = 1 the computed q is below 3e-7, so phi rounds to exactly 0.0.
#include "kernels.cuh"

namespace raattn {
namespace {

constexpr int BM = 128;   // query rows per CTA: the MMA M and the 128 TMEM lanes
constexpr int BN = 128;   // keys per tile: the N of Q K^T and the K of P V
// 16 softmax warps, four per scheduler: warps w, w + 4, w + 8, w + 12 share TMEM lanes
// 32 (w % 4) .. + 31 (the same query rows) and split each tile's 128 key columns into
// NPART parts of WCOLS.  More warps per scheduler hide the latencies of the per-score
// chain (TMEM load, FMA, reciprocal, conversion, shared-memory store).
constexpr int SOFTMAX_WARPS = 8;
constexpr int NPART = SOFTMAX_WARPS / 4;
constexpr int WCOLS = 128 / NPART;
constexpr int PRODUCER_WARP = SOFTMAX_WARPS;
constexpr int MMA_WARP = SOFTMAX_WARPS + 1;
constexpr int THREADS = 32 * (SOFTMAX_WARPS + 2);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S0 = 0;
constexpr uint32_t TMEM_S1 = 128;
constexpr uint32_t TMEM_O = 256;
constexpr int BOX_BYTES = 128 * 64 * 2;   // one TMA box: 128 rows x 64 bf16 (128 B per row)

template <int D>
struct FwdCfg {
  static constexpr int TILE_BYTES = BN * D * 2;   // a Q, K or V tile: D/64 boxes
  // Ring depth: enough K/V tiles in flight to cover the L2 -> shared-memory TMA latency
  // at one tile consumed per ~512 tensor cycles.
  static constexpr int NSTAGE = (D == 128) ? 4 : 8;
  static constexpr int P_BYTES = BM * BN * 2;     // P tile: two 64-key halves of 16 KB
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + TILE_BYTES;
  static constexpr int OFF_P = OFF_RING + NSTAGE * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  // q_full, ring_full[NSTAGE], ring_empty[NSTAGE], s_full[2], s_empty[2], p_full[2], p_empty[2], o_full, drain
  static constexpr int NUM_BARS = 1 + 2 * NSTAGE + 8 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int MISC_BYTES = 16 + 2 * SOFTMAX_WARPS * 4;   // tmem base, abort flag, live votes
  static constexpr int OFF_XCH = OFF_MISC + MISC_BYTES;   // [NPART][128] floats + [NPART][128] ints
  static constexpr int USED = OFF_XCH + 2 * NPART * BM * 4;
  // alignment slack only where it fits; otherwise the kernel requires (and checks) a
  // 1024-byte aligned dynamic shared-memory base
  static constexpr int SLACK = (USED + 1024 <= 232448) ? 1024 : 0;
  static constexpr int SMEM_BYTES = USED + SLACK;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// phi for two scores of a row: w = sat(base - c2 s) = (1+u)/2, one reciprocal for the pair
// (R = 1/(w0 w1), so 1/w0 = R w1), q = 1/w - 1 as a single FMA, phi = ((q^2)^2)^2 in f32x2.
__device__ __forceinline__ float2 phi_pair(float s0, float s1, float c2, float base) {
  const float w0 = fma_sat(s0, -c2, base);
  const float w1 = fma_sat(s1, -c2, base);
  const float R = rcp_approx(w0 * w1);
  const float2 qq = make_float2(fmaf(R, w1, -1.0f), fmaf(R, w0, -1.0f));
  const float2 q2 = __fmul2_rn(qq, qq);
  const float2 q4 = __fmul2_rn(q2, q2);
  return __fmul2_rn(q4, q4);
}

// Pass-2 work of one WCOLS-column part of a tile: phi, the fp16 P chunks in the swizzled
// tile, and the partial row sum.  MASKED: columns past `lim` (causal diagonal, ragged
// tail) get s = -inf, hence w = 1 and phi = 0.
template <bool MASKED>
__device__ __forceinline__ float2 pass2_part_tile(const uint32_t (&sv)[WCOLS / 32][32], uint8_t* prow,
                                                  int row_local, int cbase, int col0, int lim, float c2,
                                                  float base) {
  float2 tsum2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int c8 = 0; c8 < WCOLS / 8; ++c8) {
    uint32_t packed[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = c8 * 8 + 2 * e;
      float s0 = __uint_as_float(sv[c >> 5][c & 31]);
      float s1 = __uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]);
      if (MASKED) {
        if (col0 + c > lim) s0 = -INFINITY;
        if (col0 + c + 1 > lim) s1 = -INFINITY;
      }
      const float2 ph = phi_pair(s0, s1, c2, base);
      tsum2 = __fadd2_rn(tsum2, ph);
      packed[e] = pack_f16x2_sat(ph.x, ph.y);
    }
    const int chunk = (cbase >> 3) + c8;   // 16-byte chunk of the 128-key row
    *reinterpret_cast<uint4*>(prow + (chunk >> 3) * BOX_BYTES + (((chunk & 7) ^ (row_local & 7)) << 4)) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  return tsum2;
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }


template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_tc_kernel(const AttnShape s, const __grid_constant__ FwdTcArgs args, const LaunchCtx ctx) {
  using C = FwdCfg<D>;
  constexpr int NST = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  if (C::SLACK == 0 && mis != 0) {   // uniform across the CTA: nothing launched yet
    if (threadIdx.x == 0) atomicOr(ctx.status, kStatusBadSmem);
    return;
  }
  uint8_t* smem = smem_raw + ((1024u - mis) & 1023u);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sRing = smem + C::OFF_RING;
  uint8_t* sP = smem + C::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* ring_full = bars + 1;
  uint64_t* ring_empty = ring_full + NST;
  uint64_t* s_full = ring_empty + NST;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 2;
  uint64_t* o_full = p_empty + 2;
  uint64_t* drain = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* live = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);   // [2][8]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BH = s.B * s.H;
  const int nqt = (s.NQ + BM - 1) / BM;
  const int item = blockIdx.x;
  // Head-major order: the ~150 resident CTAs share a few heads, so each head's K and V
  // (4 MB at N = 8192, D = 128) stay in L2 across its query tiles.  Causal: within a
  // head the longest query tiles (largest index) go first.
  const int bh = item / nqt;
  const int qt = s.causal ? (nqt - 1 - item % nqt) : (item % nqt);
  const int q0 = qt * BM;
  const int last_key = s.causal ? min(s.NK - 1, min(s.NQ - 1, q0 + BM - 1)) : s.NK - 1;
  const int nkt = last_key / BN + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], SOFTMAX_WARPS);   // one arrival per softmax warp
      mbar_init(&p_full[i], SOFTMAX_WARPS);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&args.tm_q);
      tma_prefetch_desc(&args.tm_k);
      tma_prefetch_desc(&args.tm_v);
      mbar_arrive_expect_tx(q_full, C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * BOX_BYTES, &args.tm_q, q_full, c * 64, q0, bh);
      uint32_t it = 0;
      uint32_t last_par[NST];
      bool issued[NST];
#pragma unroll
      for (int i = 0; i < NST; ++i) {
        issued[i] = false;
        last_par[i] = 0;
      }
      auto issue = [&](const CUtensorMap* map, int j) -> bool {
        const int st = it % NST;
        const uint32_t par = (it / NST) & 1u;
        if (!mbar_wait(&ring_empty[st], par ^ 1u, abort_flag, ctx)) return false;
        mbar_arrive_expect_tx(&ring_full[st], C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sRing + st * C::TILE_BYTES + c * BOX_BYTES, map, &ring_full[st], c * 64, j * BN, bh);
        issued[st] = true;
        last_par[st] = par;
        ++it;
        return true;
      };
      bool ok = true;
      for (int j = 0; j < nkt && ok; ++j) ok = issue(&args.tm_k, j);         // pass 1: K_0 .. K_{n-1}
      if (ok) ok = issue(&args.tm_k, 0);                                     // pass 2: K_0, then
      for (int j = 1; j < nkt && ok; ++j) {                                  //   K_j, V_{j-1}
        ok = issue(&args.tm_k, j);
        if (ok) ok = issue(&args.tm_v, j - 1);
      }
      if (ok) ok = issue(&args.tm_v, nkt - 1);                               //   V_{n-1}
      drain_wait(q_full, 0, ctx);
      for (int i = 0; i < NST; ++i)
        if (issued[i]) drain_wait(&ring_full[i], last_par[i], ctx);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_fp16_f32(BM, D, 0, 1);   // P and V in fp16
      const uint32_t sQa = smem_u32(sQ), sRa = smem_u32(sRing), sPa = smem_u32(sP);
      uint32_t it = 0, sidx = 0;
      unsigned long long visited = 0, skipped = 0;
      bool o_started = false;
      auto mma_s = [&]() -> bool {   // S[sidx & 1] = Q K^T, K from ring slot `it`
        const int st = it % NST;
        const uint32_t par = (it / NST) & 1u;
        const int sb = sidx & 1;
        const uint32_t spar = (sidx >> 1) & 1u;
        if (!mbar_wait(&ring_full[st], par, abort_flag, ctx)) return false;
        if (!mbar_wait(&s_empty[sb], spar ^ 1u, abort_flag, ctx)) return false;
        tc_fence_after();
        const uint32_t kaddr = sRa + st * C::TILE_BYTES;
        const uint32_t dcol = tmem + (sb ? TMEM_S1 : TMEM_S0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;
          tc_mma_f16(dcol, smem_desc_sw128(sQa + off, 16, 1024), smem_desc_sw128(kaddr + off, 16, 1024),
                     idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&ring_empty[st]);
        tc_commit(&s_full[sb]);
        ++it;
        ++sidx;
        return true;
      };
      auto mma_pv = [&](int t) -> bool {   // O += P_t V_t, V from ring slot `it`
        const int pb = t & 1;
        const uint32_t ppar = (t >> 1) & 1u;
        const int st = it % NST;
        if (!mbar_wait(&p_full[pb], ppar, abort_flag, ctx)) return false;
        if (!mbar_wait(&ring_full[st], (it / NST) & 1u, abort_flag, ctx)) return false;
        tc_fence_after();
        int any = 0;
#pragma unroll
        for (int w = 0; w < SOFTMAX_WARPS; ++w) any |= live[pb * SOFTMAX_WARPS + w];
        const bool is_live = any != 0;
        ++visited;
        if (is_live) {
          const uint32_t vaddr = sRa + st * C::TILE_BYTES;
          const uint32_t paddr = sPa + pb * C::P_BYTES;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t aoff = (kk >> 2) * BOX_BYTES + (kk & 3) * 32;   // P: K-major, 16 keys = 32 B
            const uint32_t boff = kk * 16 * 128;                            // V: MN-major, 16 key rows
            tc_mma_f16(tmem + TMEM_O, smem_desc_sw128(paddr + aoff, 16, 1024),
                       smem_desc_sw128(vaddr + boff, BOX_BYTES, 1024), idesc_pv,
                       (o_started || kk > 0) ? 1u : 0u);
          }
          o_started = true;
        } else {
          ++skipped;
        }
        tc_commit(&ring_empty[st]);
        tc_commit(&p_empty[pb]);
        ++it;
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, ctx);
      // test knob: nothing is committed to `drain` yet, so this wait can only time out
      if (ok && ctx.force_timeout) ok = mbar_wait(drain, 0, abort_flag, ctx);
      for (int j = 0; j < nkt && ok; ++j) ok = mma_s();   // pass 1
      if (ok) ok = mma_s();                                // pass 2
      for (int j = 1; j < nkt && ok; ++j) {
        ok = mma_s();
        if (ok) ok = mma_pv(j - 1);
      }
      if (ok) ok = mma_pv(nkt - 1);
      if (ok) tc_commit(o_full);
      tc_commit(drain);
      drain_wait(drain, 0, ctx);
      if (ok && args.tile_counts) {
        atomicAdd(&args.tile_counts[0], visited);
        atomicAdd(&args.tile_counts[1], skipped);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31 (query rows) and key columns
    // [WCOLS (w / 4), WCOLS (w / 4) + WCOLS) of every tile; the row maximum, its argmax
    // and the row sum are combined across the NPART parts through shared memory.
    const int quarter = warp & 3;
    const int part = warp >> 2;
    const int cbase = part * WCOLS;
    const int row_local = quarter * 32 + lane;   // TMEM lane
    const int row = q0 + row_local;
    const int lim = s.causal ? min(row, s.NK - 1) : s.NK - 1;   // last key this row may see
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* xf = reinterpret_cast<float*>(smem + C::OFF_XCH);              // [NPART][BM]
    int* xi = reinterpret_cast<int*>(smem + C::OFF_XCH + NPART * BM * 4);  // [NPART][BM]
    auto group_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(32 * SOFTMAX_WARPS) : "memory"); };
    auto warp_wait = [&](uint64_t* bar, uint32_t par) -> bool {
      int r = 1;
      if (lane == 0) r = mbar_wait(bar, par, abort_flag, ctx) ? 1 : 0;
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    uint32_t sv[WCOLS / 32][32];
    auto load_s = [&](int sb) {
      const uint32_t col = lane_addr + (sb ? TMEM_S1 : TMEM_S0) + cbase;
#pragma unroll
      for (int k = 0; k < WCOLS / 32; ++k) tmem_ld32(col + 32 * k, sv[k]);
      tc_wait_ld();
    };
#define SV(c) u2f(sv[(c) >> 5][(c) & 31])

    bool ok = true;
    uint32_t sidx = 0;
    float m = -INFINITY;
    int a = -1;
    // pass 1: running maximum of the raw scores q.k over this part's columns (scale > 0
    // keeps the argmax)
    for (int j = 0; j < nkt && ok; ++j) {
      const int sb = sidx & 1;
      const uint32_t spar = (sidx >> 1) & 1u;
      ok = warp_wait(&s_full[sb], spar);
      if (!ok) break;
      tc_fence_after();
      load_s(sb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[sb]);
      ++sidx;
      const int col0 = j * BN + cbase;   // key index of local column 0
      const bool need_mask = col0 + WCOLS - 1 > lim;
      float t0 = -INFINITY, t1 = -INFINITY, t2 = -INFINITY, t3 = -INFINITY;
      if (!need_mask) {
#pragma unroll
        for (int c = 0; c < WCOLS; c += 8) {
          t0 = max3f(t0, SV(c), SV(c + 1));
          t1 = max3f(t1, SV(c + 2), SV(c + 3));
          t2 = max3f(t2, SV(c + 4), SV(c + 5));
          t3 = max3f(t3, SV(c + 6), SV(c + 7));
        }
      } else {
#pragma unroll
        for (int c = 0; c < WCOLS; ++c) {
          const float x = (col0 + c <= lim) ? SV(c) : -INFINITY;
          if ((c & 3) == 0) t0 = fmaxf(t0, x);
          if ((c & 3) == 1) t1 = fmaxf(t1, x);
          if ((c & 3) == 2) t2 = fmaxf(t2, x);
          if ((c & 3) == 3) t3 = fmaxf(t3, x);
        }
      }
      const float tmax = fmaxf(fmaxf(t0, t1), fmaxf(t2, t3));
      if (tmax > m) {   // strictly greater: an earlier tile keeps ties (lowest index)
        int idx = WCOLS;
#pragma unroll
        for (int c = WCOLS - 1; c >= 0; --c)
          if (SV(c) == tmax && col0 + c <= lim) idx = c;
        m = tmax;
        a = col0 + idx;
      }
    }
    // combine the parts (reached by every softmax warp, also after a wait gave up): the
    // maximum, and among the parts that attain it the lowest index
    xf[part * BM + row_local] = m;
    xi[part * BM + row_local] = a;
    group_sync();
    m = xf[row_local];
#pragma unroll
    for (int p = 1; p < NPART; ++p) m = fmaxf(m, xf[p * BM + row_local]);
    a = -1;
#pragma unroll
    for (int p = 0; p < NPART; ++p) {
      const int ap = xi[p * BM + row_local];
      if (xf[p * BM + row_local] == m && ap >= 0 && (a < 0 || ap < a)) a = ap;
    }
    group_sync();   // xf is reused for the row sum

    // pass 2: phi, sum(phi), P tiles
    const float m_sc = m * s.scale;
    const float c2 = s.scale * (1.0f / 32.0f);
    const float base = fmaf(m_sc, 1.0f / 32.0f, 0.5f);
    float rowsum = 0.0f;
    for (int j = 0; j < nkt && ok; ++j) {
      const int sb = sidx & 1;
      const uint32_t spar = (sidx >> 1) & 1u;
      ok = warp_wait(&s_full[sb], spar);
      if (!ok) break;
      tc_fence_after();
      load_s(sb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[sb]);
      ++sidx;
      const int col0 = j * BN + cbase;
      const bool need_mask = col0 + WCOLS - 1 > lim;
      const int pb = j & 1;
      ok = warp_wait(&p_empty[pb], ((j >> 1) & 1u) ^ 1u);
      if (!ok) break;
      uint8_t* prow = sP + pb * C::P_BYTES + row_local * 128;
      const float2 tsum2 = need_mask ? pass2_part_tile<true>(sv, prow, row_local, cbase, col0, lim, c2, base)
                                     : pass2_part_tile<false>(sv, prow, row_local, cbase, col0, lim, c2, base);
      fence_proxy_async_smem();
      const float tsum = tsum2.x + tsum2.y;
      const unsigned any_live = __any_sync(0xffffffffu, tsum > 0.0f);
      if (lane == 0) live[pb * SOFTMAX_WARPS + warp] = any_live ? 1 : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
      rowsum += tsum;
    }
#undef SV
    xf[part * BM + row_local] = rowsum;
    group_sync();
    rowsum = xf[row_local];
#pragma unroll
    for (int p = 1; p < NPART; ++p) rowsum += xf[p * BM + row_local];
    if (ok) ok = warp_wait(o_full, 0);
    if (ok) {
      tc_fence_after();
      const bool row_ok = row < s.NQ;
      const float inv = 1.0f / rowsum;
      const size_t ro = static_cast<size_t>(bh) * s.NQ + (row_ok ? row : 0);
      // the parts store 32-column slices of the D output columns of their rows
#pragma unroll
      for (int c0 = part * 32; c0 < D; c0 += NPART * 32) {
        uint32_t ov[32];
        tmem_ld32(lane_addr + TMEM_O + c0, ov);
        tc_wait_ld();
        if (row_ok) {
          if (args.out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(args.o) + ro * D + c0);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 pk;
              pk.x = pack_bf16x2(u2f(ov[v4 * 8 + 0]) * inv, u2f(ov[v4 * 8 + 1]) * inv);
              pk.y = pack_bf16x2(u2f(ov[v4 * 8 + 2]) * inv, u2f(ov[v4 * 8 + 3]) * inv);
              pk.z = pack_bf16x2(u2f(ov[v4 * 8 + 4]) * inv, u2f(ov[v4 * 8 + 5]) * inv);
              pk.w = pack_bf16x2(u2f(ov[v4 * 8 + 6]) * inv, u2f(ov[v4 * 8 + 7]) * inv);
              dst[v4] = pk;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(args.o) + ro * D + c0);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(u2f(ov[v4 * 4 + 0]) * inv, u2f(ov[v4 * 4 + 1]) * inv,
                                    u2f(ov[v4 * 4 + 2]) * inv, u2f(ov[v4 * 4 + 3]) * inv);
          }
        }
      }
      if (row_ok && part == 0) {
        if (args.row_m) args.row_m[ro] = m_sc;
        if (args.row_s) args.row_s[ro] = rowsum;
        if (args.row_arg) args.row_arg[ro] = a;
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_fwd_d(const AttnShape& s, const FwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st) {
  using C = FwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int nqt = (s.NQ + BM - 1) / BM;
  const unsigned grid = static_cast<unsigned>(nqt) * static_cast<unsigned>(s.B * s.H);
  attn_fwd_tc_kernel<D><<<grid, THREADS, C::SMEM_BYTES, st>>>(s, a, ctx);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_tc(const AttnShape& s, const FwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st) {
  if (s.D == 128) return launch_fwd_d<128>(s, a, ctx, st);
  if (s.D == 64) return launch_fwd_d<64>(s, a, ctx, st);
  return cudaErrorInvalidValue;
}

}  // namespace raattn
