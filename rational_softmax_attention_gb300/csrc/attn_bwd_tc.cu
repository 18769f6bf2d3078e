// bf16 ra_attention backward on the tensor cores (tcgen05 + TMEM + TMA).
//
// Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax
// "Closed-Form Backward Pass": d phi/du = -16 phi/(1-u^2), evaluated from the
// recomputed u and p, with no saved powers of q; section 3, ra_attention:
// "tiled forward and backward" keeping only O(B H N_Q D) saved state (O and the
// per-row max, sum and argmax of the forward).
//
// Chain rule (the gradient of x_max goes to the lowest-index argmax a_i):
//   P = phi / s_i,  dP = dO V^T,  D_i = dO_i . O_i,
//   E_ij = P_ij (dP_ij - D_i) / (1 - u_ij^2)   for allowed j != a_i with u_ij < 1,
//   R_i = sum_j E_ij,   dS = E with dS_{i,a_i} = -R_i,
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// With w = (1+u)/2 and q = 1/w - 1:  phi/(1-u^2) = q^7 / (4 w^2),  so
//   E_ij = [q^7 (1/w)^2 / (4 s_i)] (dP_ij - D_i).
//
// Two kernels, no atomics:
//   dQ kernel (one CTA per 128-row query tile, loop over key tiles): S = Q K^T and
//     dP = dO V^T in TMEM; the softmax warpgroup (thread = query row) forms E,
//     zeroes it at the argmax, sums R_i, and writes E (bf16) to shared memory;
//     dQ += E K accumulates in TMEM; epilogue dq = scale (dQ - R_i K_{a_i}).  It
//     also writes D_i, R_i and two per-row constants to the workspace.
//   dK/dV kernel (one CTA per 128-key tile, loop over query tiles): S^T = K Q^T
//     and dP^T = V dO^T in TMEM; the softmax warpgroup (thread = key row) forms
//     P^T and dS^T (with -R_i at the argmax entries) in shared memory;
//     dV += P^T dO and dK += dS^T Q accumulate in TMEM.
// The second kernel reads what the first wrote, so they run in stream order.
//
// Operand format: the MMAs of the backward take fp16 operands (fp32 accumulation).
// A prologue converts Q, K, V and dO from bf16 to fp16 into the workspace; that is
// exact for 2^-14 <= |x| <= 65504 (bf16 has 8 significant bits, fp16 11), so for such
// operands the recomputed scores equal the forward's (smaller ones are rounded to the fp16
// subnormal spacing 2^-24), while P, E and dS -- formed in fp32 -- are rounded to
// fp16 (unit roundoff 2^-11) instead of bf16 (2^-8) before their products.  With
// |E| up to ~10 at wide score spreads, bf16 rounding alone costs ~2e-2 in dQ.
#include "kernels.cuh"
#include "phi.cuh"

namespace raattn {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BOX_BYTES = 128 * 64 * 2;


// 16-byte chunk `chunk` (0..15) of row r of a 128 x 128 bf16 K-major operand tile,
// stored as two 64-column halves in the 128-byte-swizzled layout TMA and tcgen05 use.
__device__ __forceinline__ void st_tile16(uint8_t* tile, int r, int chunk, uint4 val) {
  const int half = chunk >> 3, c = chunk & 7;
  *reinterpret_cast<uint4*>(tile + half * BOX_BYTES + r * 128 + ((c ^ (r & 7)) << 4)) = val;
}

// The backward coefficient q^7 (1/w)^2 for four scores x of a row, w = sat(base - c2 x) =
// (1+u)/2, q = 1/w - 1.  Four entries share two reciprocals: with the pairs A = (w0, w1),
// B = (w2, w3), R = 1/(A B) elementwise gives R B = (1/w0, 1/w1) and R A = (1/w2, 1/w3).
__device__ __forceinline__ float2 coef_pair(float2 rw) {   // rw = 1/w for two entries
  const float2 q = __fadd2_rn(rw, make_float2(-1.0f, -1.0f));
  const float2 q2 = __fmul2_rn(q, q);
  const float2 q4 = __fmul2_rn(q2, q2);
  const float2 q7 = __fmul2_rn(__fmul2_rn(q4, q2), q);
  return __fmul2_rn(q7, __fmul2_rn(rw, rw));
}
__device__ __forceinline__ void coef_quad(const float (&x)[4], float c2, float base, float2& ca, float2& cb) {
  const float2 A = make_float2(fma_sat(x[0], -c2, base), fma_sat(x[1], -c2, base));
  const float2 B = make_float2(fma_sat(x[2], -c2, base), fma_sat(x[3], -c2, base));
  const float2 P = __fmul2_rn(A, B);
  const float2 R = make_float2(rcp_approx(P.x), rcp_approx(P.y));
  ca = coef_pair(__fmul2_rn(R, B));
  cb = coef_pair(__fmul2_rn(R, A));
}

// Row of 8 bf16 from global memory as floats.
__device__ __forceinline__ void load8_bf16(const void* p, float* out) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

// ============================================================================ dQ kernel
template <int D>
struct DqCfg {
  static constexpr int TILE = BN * D * 2;
  static constexpr int NKS = 3;                    // K stages: K_j lives from S_j to dQ_j
  static constexpr int NVS = 2;                    // V stages
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TILE;
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NKS * TILE;
  static constexpr int OFF_BAR = OFF_V + NVS * TILE;
  // qdo_full, k_full[NKS], k_empty[NKS], v_full[NVS], v_empty[NVS], s_full[2], e_free[2],
  // dp_full, dp_free, e_full[2], dq_full, drain[2]
  static constexpr int NUM_BARS = 1 + 2 * NKS + 2 * NVS + 11;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_XCH = OFF_MISC + 16;   // [4][128] floats: per-part partials of D_i, then R_i
  static constexpr int USED = OFF_XCH + 4 * BM * 4;
  // alignment slack only where it fits; otherwise the kernel requires (and checks) a
  // 1024-byte aligned dynamic shared-memory base
  static constexpr int SLACK = (USED + 1024 <= 232448) ? 1024 : 0;
  static constexpr int SMEM_BYTES = USED + SLACK;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(OFF_BAR - OFF_K >= 16 * 4096, "epilogue staging: 4 KB per softmax warp in the K/V stages");
};
constexpr uint32_t DQ_TM_S0 = 0, DQ_TM_S1 = 128, DQ_TM_DP = 256, DQ_TM_DQ = 384;
// 16 softmax warps, four per scheduler: warp w owns TMEM lanes 32 (w % 4) .. + 31 (its query
// rows) and key columns [32 (w / 4), 32 (w / 4) + 32) of every tile.
constexpr int DQ_SOFTMAX_WARPS = 16;
constexpr int DQ_COLS = BN * 4 / DQ_SOFTMAX_WARPS;   // 32
constexpr int DQ_PARTS = DQ_SOFTMAX_WARPS / 4;       // warps sharing a row quarter
constexpr int DQ_PRODUCER_WARP = DQ_SOFTMAX_WARPS;
// two MMA-issuing threads: the first issues S and dP, the second dQ.  A barrier wait
// stalls its issuing thread for a few hundred cycles, longer than the two 64-cycle
// products the tensor queue holds; the other issuer's products fill that time.
constexpr int DQ_MMA_WARP = DQ_SOFTMAX_WARPS + 1;
constexpr int DQ_THREADS = 32 * (DQ_SOFTMAX_WARPS + 3);
static_assert(DQ_COLS == 32, "one 32-column TMEM load per softmax warp and tile");

__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(DQ_SOFTMAX_WARPS * 32) : "memory");
}

// MASK: a boolean attention mask (args.mask_q, rows = queries) applies on top of `causal`.
// nk: the keys taken, N_K, or fewer for a query tile run as an unmasked one over the keys its
// mask leaves (the per-row plain lengths of the tile maps).
template <int D, bool MASK>
__device__ __forceinline__ void dq_body(const AttnShape& s, const BwdTcArgs& args, const LaunchCtx& ctx, int nk) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  if (C::SLACK == 0 && mis != 0) {   // uniform across the CTA: nothing launched yet
    if (threadIdx.x == 0) atomicOr(ctx.status, kStatusBadSmem);
    return;
  }
  uint8_t* smem = smem_raw + ((1024u - mis) & 1023u);
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* qdo_full = bars;
  uint64_t* k_full = qdo_full + 1;
  uint64_t* k_empty = k_full + C::NKS;
  uint64_t* v_full = k_empty + C::NKS;
  uint64_t* v_empty = v_full + C::NVS;
  uint64_t* s_full = v_empty + C::NVS;
  // e_free[b]: the dQ product has read E from score buffer b (E_j is written over S_j)
  uint64_t* e_free = s_full + 2;
  uint64_t* dp_full = e_free + 2;
  uint64_t* dp_free = dp_full + 1;
  // e_full[b]: every softmax warp has written E into score buffer b.  One barrier per
  // buffer: a warp that has finished tile j may finish tile j + 1 (dP_{j+1} waits only for
  // dp_free) before a slower warp's arrival for tile j, but never tile j + 2 (S_{j+2} waits
  // for the dQ product of tile j), so arrivals for consecutive tiles never share a phase.
  uint64_t* e_full = dp_free + 1;
  uint64_t* dq_full = e_full + 2;
  uint64_t* drain = dq_full + 1;   // [2], one per issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqt = (s.NQ + BM - 1) / BM;
  const int item = blockIdx.x;
  // head-major order (K/V of a head shared in L2), longest causal query tiles first
  const int bh = item / nqt;
  const int qt = s.causal ? (nqt - 1 - item % nqt) : (item % nqt);
  const int q0 = qt * BM;
  const int last_key = s.causal ? min(nk - 1, min(s.NQ - 1, q0 + BM - 1)) : nk - 1;
  const int nkt = last_key / BN + 1;
  // Key tiles 32 w .. 32 w + 31 this query tile takes, as bits: its range and, with a tile
  // live map, the tiles holding an allowed pair.  Every role walks them in key order and
  // counts them: ring slots, score buffers and barrier phases follow that count, so a fully
  // masked tile costs nothing (no copy, no product, no arithmetic).  Unmasked: every tile.
  auto take_word = [&](int w) -> uint32_t {
    const int n = nkt - 32 * w;
    uint32_t bits = n >= 32 ? ~0u : (n > 0 ? (1u << n) - 1u : 0u);
    if constexpr (MASK) {
      if (args.mask_q.live && bits) {
        const int gm = (args.mask_q.mb > 1 ? bh / s.H : 0) * args.mask_q.mh + (args.mask_q.mh > 1 ? bh % s.H : 0);
        bits &= args.mask_q.live[(static_cast<size_t>(gm) * nqt + qt) * args.mask_q.live_words + w];
      }
    }
    return bits;
  };
  // Key tiles 32 w .. 32 w + 31 the mask allows whole to every row of this query tile: their
  // mask words are all ones and are not read.
  auto full_word = [&](int w) -> uint32_t {
    if constexpr (MASK) {
      if (args.mask_q.full) {
        const int gm = (args.mask_q.mb > 1 ? bh / s.H : 0) * args.mask_q.mh + (args.mask_q.mh > 1 ? bh % s.H : 0);
        return args.mask_q.full[(static_cast<size_t>(gm) * nqt + qt) * args.mask_q.live_words + w];
      }
    }
    return 0u;
  };

  if (threadIdx.x == 0) {
    mbar_init(qdo_full, 1);
    for (int i = 0; i < C::NKS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 2);   // S_j (issuer 0) and dQ_j (issuer 1) both read K_j
    }
    for (int i = 0; i < C::NVS; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&e_free[i], 1);
    }
    mbar_init(dp_full, 1);
    mbar_init(dp_free, DQ_SOFTMAX_WARPS);
    mbar_init(&e_full[0], DQ_SOFTMAX_WARPS);
    mbar_init(&e_full[1], DQ_SOFTMAX_WARPS);
    mbar_init(dq_full, 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == DQ_MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == DQ_PRODUCER_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&args.tm_q);
      tma_prefetch_desc(&args.tm_k);
      tma_prefetch_desc(&args.tm_v);
      tma_prefetch_desc(&args.tm_do);
      mbar_arrive_expect_tx(qdo_full, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sQ + c * BOX_BYTES, &args.tm_q, qdo_full, c * 64, q0, bh);
        tma_load_3d(sDO + c * BOX_BYTES, &args.tm_do, qdo_full, c * 64, q0, bh);
      }
      bool ok = true;
      int k_issued = 0, v_issued = 0;
      uint32_t tw = 0;
      for (int j = 0, c = 0; j < nkt && ok; ++j) {
        if constexpr (MASK) {
          if ((j & 31) == 0) tw = take_word(j >> 5);
          if (!((tw >> (j & 31)) & 1u)) continue;
        }
        const int ks = c % C::NKS;
        ok = mbar_wait(&k_empty[ks], ((c / C::NKS) & 1u) ^ 1u, abort_flag, ctx);
        if (!ok) break;
        mbar_arrive_expect_tx(&k_full[ks], C::TILE);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc)
          tma_load_3d(sK + ks * C::TILE + cc * BOX_BYTES, &args.tm_k, &k_full[ks], cc * 64, j * BN, bh);
        k_issued = c + 1;
        const int vs = c % C::NVS;
        ok = mbar_wait(&v_empty[vs], ((c / C::NVS) & 1u) ^ 1u, abort_flag, ctx);
        if (!ok) break;
        mbar_arrive_expect_tx(&v_full[vs], C::TILE);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc)
          tma_load_3d(sV + vs * C::TILE + cc * BOX_BYTES, &args.tm_v, &v_full[vs], cc * 64, j * BN, bh);
        v_issued = c + 1;
        ++c;
      }
      // drain every copy issued (the last fill of each stage)
      drain_wait(qdo_full, 0, ctx);
      for (int j = max(0, k_issued - C::NKS); j < k_issued; ++j)
        drain_wait(&k_full[j % C::NKS], (j / C::NKS) & 1u, ctx);
      for (int j = max(0, v_issued - C::NVS); j < v_issued; ++j)
        drain_wait(&v_full[j % C::NVS], (j / C::NVS) & 1u, ctx);
    }
  } else if (warp >= DQ_MMA_WARP) {
    const int who = warp - DQ_MMA_WARP;   // 0: S and dP products; 1: dQ products
    if (lane == 0) {
      constexpr uint32_t idesc_ss = idesc_fp16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_kmn = idesc_fp16_f32(BM, D, 0, 1);
      constexpr uint32_t HI = sdesc_hi_sw128(1024);
      const uint32_t qlo = sdesc_lo(smem_u32(sQ), 16), dolo = sdesc_lo(smem_u32(sDO), 16);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = mbar_wait(qdo_full, 0, abort_flag, ctx);
      // test knob: nothing is committed to `drain` yet, so this wait can only time out
      if (ok && ctx.force_timeout) ok = mbar_wait(&drain[who], 0, abort_flag, ctx);
      uint32_t tw = 0;
      if (who == 0) {
        for (int j = 0, c = 0; j < nkt && ok; ++j) {
          if constexpr (MASK) {
            if ((j & 31) == 0) tw = take_word(j >> 5);
            if (!((tw >> (j & 31)) & 1u)) continue;
          }
          // S_j = Q K_j^T, the c-th tile taken
          const int ks = c % C::NKS, sb = c & 1;
          // buffer sb is free once the dQ product of tile c - 2 has read E_{c-2} from it
          // (the softmax warps loaded S_{c-2} before writing E_{c-2})
          ok = mbar_wait(&k_full[ks], (c / C::NKS) & 1u, abort_flag, ctx) &&
               mbar_wait(&e_free[sb], ((c >> 1) & 1u) ^ 1u, abort_flag, ctx);
          if (!ok) break;
          tc_fence_after();
          const uint32_t klo = sdesc_lo(aK + ks * C::TILE, 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
            tc_mma_f16(tmem + (sb ? DQ_TM_S1 : DQ_TM_S0), sdesc(qlo + off, HI), sdesc(klo + off, HI), idesc_ss,
                       kk > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[sb]);
          tc_commit(&k_empty[ks]);
          // dP_j = dO V_j^T
          const int vs = c % C::NVS;
          ok = mbar_wait(&v_full[vs], (c / C::NVS) & 1u, abort_flag, ctx) &&
               mbar_wait(dp_free, (c & 1u) ^ 1u, abort_flag, ctx);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vlo = sdesc_lo(aV + vs * C::TILE, 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
            tc_mma_f16(tmem + DQ_TM_DP, sdesc(dolo + off, HI), sdesc(vlo + off, HI), idesc_ss, kk > 0 ? 1u : 0u);
          }
          tc_commit(&v_empty[vs]);
          tc_commit(dp_full);
          ++c;
        }
      } else {
        for (int j = 0, t = 0; j < nkt && ok; ++j) {   // dQ += E_t K_t, t counting the tiles taken
          if constexpr (MASK) {
            if ((j & 31) == 0) tw = take_word(j >> 5);
            if (!((tw >> (j & 31)) & 1u)) continue;
          }
          const int ks = t % C::NKS;
          ok = mbar_wait(&e_full[t & 1], (t >> 1) & 1u, abort_flag, ctx) &&
               mbar_wait(&k_full[ks], (t / C::NKS) & 1u, abort_flag, ctx);
          if (!ok) break;
          tc_fence_after();
          const uint32_t klo = sdesc_lo(aK + ks * C::TILE, BOX_BYTES);
          // E_t from tensor memory: fp16 pairs over the first half of each softmax warp's
          // columns of score buffer t & 1, 8 columns per 16 keys
          const uint32_t ecol = tmem + ((t & 1) ? DQ_TM_S1 : DQ_TM_S0);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            tc_mma_f16_ts(tmem + DQ_TM_DQ, ecol + (16 * kk / DQ_COLS) * DQ_COLS + (16 * kk % DQ_COLS) / 2,
                          sdesc(klo + ((kk * 2048) >> 4), HI), idesc_kmn, (t > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&k_empty[ks]);
          tc_commit(&e_free[t & 1]);
          ++t;
        }
        if (ok) tc_commit(dq_full);
      }
      tc_commit(&drain[who]);
      drain_wait(&drain[who], 0, ctx);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps (row = query)
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31 (query rows) and key columns
    // [32 (w / 4), 32 (w / 4) + 32) of every tile; D_i and R_i are combined across the
    // four parts of a row through shared memory.
    const int quarter = warp & 3;
    const int part = warp >> 2;
    const int cbase = part * DQ_COLS;
    const int r = quarter * 32 + lane;
    const int i = q0 + r;
    const bool i_ok = i < s.NQ;
    const size_t ro = static_cast<size_t>(bh) * s.NQ + (i_ok ? i : s.NQ - 1);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);   // [DQ_PARTS][BM]
    auto warp_wait = [&](uint64_t* bar, uint32_t par) -> bool {
      int okv = 1;
      if (lane == 0) okv = mbar_wait(bar, par, abort_flag, ctx) ? 1 : 0;
      return __shfl_sync(0xffffffffu, okv, 0) != 0;
    };
    const float m_sc = args.row_m[ro];
    const float row_s = args.row_s[ro];
    const float inv_s = row_s > 0.0f ? 1.0f / row_s : 0.0f;   // 0: a row with no visible key
    const int a = min(max(args.row_arg[ro], 0), s.NK - 1);
    // this row's attention-mask words: four per key tile, one per warp part
    const uint32_t* mrow = nullptr;
    if (MASK) {
      const int gm = (args.mask_q.mb > 1 ? bh / s.H : 0) * args.mask_q.mh + (args.mask_q.mh > 1 ? bh % s.H : 0);
      mrow = args.mask_q.bits + (static_cast<size_t>(gm) * s.NQ + (i_ok ? i : s.NQ - 1)) * args.mask_q.words;
    }
    // D_i = dO_i . O_i: each part of the warps sums D / DQ_PARTS of the dimensions
    {
      float acc = 0.0f;
      const char* dorow = reinterpret_cast<const char*>(args.dout) + ro * D * 2;
#pragma unroll 4
      for (int d = part * (D / DQ_PARTS); d < (part + 1) * (D / DQ_PARTS); d += 8) {
        float g[8], o[8];
        load8_bf16(dorow + d * 2, g);
        if (args.o_bf16) {
          load8_bf16(reinterpret_cast<const char*>(args.o) + (ro * D + d) * 2, o);
        } else {
          const float4* op = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(args.o) + ro * D + d);
          const float4 x0 = op[0], x1 = op[1];
          o[0] = x0.x; o[1] = x0.y; o[2] = x0.z; o[3] = x0.w;
          o[4] = x1.x; o[5] = x1.y; o[6] = x1.z; o[7] = x1.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(g[e], o[e], acc);
      }
      xch[part * BM + r] = acc;
    }
    softmax_sync();
    float Di = 0.0f;
#pragma unroll
    for (int pp = 0; pp < DQ_PARTS; ++pp) Di += xch[pp * BM + r];
    softmax_sync();   // xch is reused for R_i after the loop
    // rows past N_Q read zero-filled Q rows (s = 0): base 2 saturates every w to 1, weight 0
    const float base = (i_ok && m_sc > -INFINITY) ? fmaf(m_sc, 1.0f / 32.0f, 0.5f) : 2.0f;
    const float c2 = s.scale * (1.0f / 32.0f);
    const float cE = 0.25f * inv_s;
    const int lim = s.causal ? min(i, nk - 1) : nk - 1;
    const float2 cE2 = make_float2(cE, cE), mcED2 = make_float2(-cE * Di, -cE * Di);
    float2 R2 = make_float2(0.0f, 0.0f);
    bool ok = true;
    uint32_t sv[32];
#define SV(c) sv[c]
    uint32_t tw = 0, fw = 0;
    int ntaken = 0;   // key tiles taken (their E written); 0 leaves the dQ accumulator unwritten
    for (int j = 0; j < nkt && ok; ++j) {
      if constexpr (MASK) {
        if ((j & 31) == 0) {
          tw = take_word(j >> 5);
          fw = full_word(j >> 5);
        }
        if (!((tw >> (j & 31)) & 1u)) continue;
      }
      const int cnt = ntaken++;
      const int sb = cnt & 1;
      // in flight during the wait; a tile the mask allows whole reads none
      const uint32_t mw = (MASK && !((fw >> (j & 31)) & 1u)) ? mrow[4 * j + part] : ~0u;
      ok = warp_wait(&s_full[sb], (cnt >> 1) & 1u);
      if (!ok) break;
      tc_fence_after();
      {
        const uint32_t col = lane_addr + (sb ? DQ_TM_S1 : DQ_TM_S0) + cbase;
        tmem_ld32(col, sv);
        tc_wait_ld();
      }
      const int col0 = j * BN + cbase;   // key index of local column 0
      // With an attention mask, a chunk every row of the warp sees whole needs no per-entry
      // test, and a chunk no row sees has zero coefficients and E (no arithmetic).  The vote
      // runs in the masked instance only, where the whole warp is here together.
      int kind = kChunkMixed;
      if constexpr (MASK) kind = chunk_kind(mw, col0, lim);
      const bool need_mask = MASK ? kind == kChunkMixed : col0 + DQ_COLS - 1 > lim;
      const bool dead = MASK && kind == kChunkNone;
      // coefficient q^7 (1/w)^2 per entry, in place; the factor 1/(4 s_i) is applied with
      // dP - D_i below.  Four entries share two reciprocals (coef_quad).
      if (dead) {
#pragma unroll
        for (int c = 0; c < DQ_COLS; ++c) SV(c) = 0u;
      }
#pragma unroll
      for (int c = 0; c < DQ_COLS && !dead; c += 4) {
        float x[4] = {u2f(SV(c)), u2f(SV(c + 1)), u2f(SV(c + 2)), u2f(SV(c + 3))};
        if (need_mask) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (col0 + c + t > lim || (MASK && !((mw >> (c + t)) & 1u))) x[t] = -INFINITY;
        }
        float2 ca, cb;
        coef_quad(x, c2, base, ca, cb);
        SV(c) = __float_as_uint(ca.x);
        SV(c + 1) = __float_as_uint(ca.y);
        SV(c + 2) = __float_as_uint(cb.x);
        SV(c + 3) = __float_as_uint(cb.y);
      }
      if (a >= col0 && a < col0 + DQ_COLS) {   // the argmax entry takes -R_i, not E
#pragma unroll
        for (int c = 0; c < DQ_COLS; ++c)
          if (col0 + c == a) SV(c) = 0u;
      }
      ok = warp_wait(dp_full, cnt & 1u);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < DQ_COLS / 32; ++cc) {
        uint32_t dv[32];
        tmem_ld32(lane_addr + DQ_TM_DP + cbase + cc * 32, dv);
        tc_wait_ld();
        if (cc == DQ_COLS / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dp_free);
        }
        // E = coef (dP - D_i) / (4 s_i) = coef (cE dP - cE D_i), as fp16 pairs over the first
        // half of this warp's (already read) columns of score buffer sb
        uint32_t e16[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          if (dead) {
            e16[t] = 0u;
            continue;
          }
          const int c = cc * 32 + 2 * t;
          const float2 dpp = make_float2(u2f(dv[2 * t]), u2f(dv[2 * t + 1]));
          const float2 ee = __fmul2_rn(make_float2(u2f(SV(c)), u2f(SV(c + 1))), __ffma2_rn(dpp, cE2, mcED2));
          R2 = __fadd2_rn(R2, ee);
          e16[t] = pack_f16x2_sat(ee.x, ee.y);
        }
        tmem_st16(lane_addr + (sb ? DQ_TM_S1 : DQ_TM_S0) + cbase + 16 * cc, e16);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&e_full[sb]);
    }
#undef SV
    // R_i over the parts (reached by every softmax warp, also after a wait gave up)
    xch[part * BM + r] = R2.x + R2.y;
    softmax_sync();
    float R = 0.0f;
#pragma unroll
    for (int pp = 0; pp < DQ_PARTS; ++pp) R += xch[pp * BM + r];
    if (ok) ok = warp_wait(dq_full, 0);
    if (ok) {
      tc_fence_after();
      if (part == 0) {   // this query tile's constant block for the dK/dV kernel
        float* blk = args.ws_consts + (static_cast<size_t>(bh) * nqt + qt) * kConstBlockFloats;
        blk[r] = base;   // 2 past N_Q: w = 1, zero weight
        blk[BM + r] = i_ok ? inv_s : 0.0f;
        blk[2 * BM + r] = i_ok ? 0.25f * Di : 0.0f;
        blk[3 * BM + r] = i_ok ? R : 0.0f;
        reinterpret_cast<int*>(blk)[4 * BM + r] = i_ok ? args.row_arg[ro] : -1;
      }
      const char* krow = reinterpret_cast<const char*>(args.k_raw) + (static_cast<size_t>(bh) * s.NK + a) * D * 2;
      // the warps of a row quarter store 32-column chunks of its rows in turn, through
      // 4 KB per warp of the K/V stages (free: dq_full means every product has completed)
      uint8_t* stage = sK + warp * 4096;
      const int wrow0 = q0 + quarter * 32;   // first row of this warp
      const size_t row0 = static_cast<size_t>(bh) * s.NQ + wrow0;
      const int n_ok = max(0, min(32, s.NQ - wrow0));
#pragma unroll
      for (int c0 = part * 32; c0 < D; c0 += 32 * DQ_PARTS) {
        uint32_t acc[32];
        tmem_ld32(lane_addr + DQ_TM_DQ + c0, acc);
        tc_wait_ld();
        float out[32];
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float kv[8];
          load8_bf16(krow + (c0 + e) * 2, kv);
#pragma unroll
          for (int t = 0; t < 8; ++t) out[e + t] = s.scale * fmaf(-R, kv[t], ntaken > 0 ? u2f(acc[e + t]) : 0.0f);
        }
        if (args.grad_bf16)
          warp_store_block32<true>(stage, out, args.dq, row0, D, c0, n_ok, lane);
        else
          warp_store_block32<false>(stage, out, args.dq, row0, D, c0, n_ok, lane);
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == DQ_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ============================================================================ dK/dV kernel
template <int D>
struct DkvCfg {
  static constexpr int TILE = BN * D * 2;
  static constexpr int NQS = 2;                    // Q stages
  static constexpr int NDS = 2;                    // dO stages
  static constexpr int A_BYTES = BN * BM * 2;      // dS^T tile (keys x queries, fp16)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NQS * TILE;
  static constexpr int OFF_DS = OFF_DO + NDS * TILE;
  // Per-query constants of one query tile, in two single-buffered parts with their own
  // lifetimes: X (base_i, 1/s_i) is read in the P^T loop, Y (D_i/4, R_i, a_i) in the dS^T
  // loop and the argmax fix-up.  X of the next tile arrives while the warps are in the
  // dS^T loop, Y while they are in the next P^T loop.  Each copy completes on the barrier
  // the softmax warps wait on anyway (X with S^T on st_full, Y with dP^T on dpt_full), so
  // a tile costs them two waits.
  static constexpr int OFF_CX = OFF_DS + A_BYTES;
  static constexpr int CX_BYTES = 2 * BM * 4;
  static constexpr int OFF_CY = OFF_CX + CX_BYTES;
  static constexpr int CY_BYTES = 3 * BM * 4;
  static constexpr int OFF_BAR = OFF_CY + CY_BYTES;
  // kv_full, q_full[NQS], q_empty[NQS], do_full[NDS], do_empty[NDS],
  // st_full, dpt_full, dpt_free, p_full[2], p_free, acc_full, drain[2],
  // cx_empty, cy_empty, ds_full, ds_free
  static constexpr int NUM_BARS = 1 + 2 * NQS + 2 * NDS + 13;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int USED = OFF_MISC + 16;
  // alignment slack only where it fits; otherwise the kernel requires (and checks) a
  // 1024-byte aligned dynamic shared-memory base
  static constexpr int SLACK = (USED + 1024 <= 232448) ? 1024 : 0;
  static constexpr int SMEM_BYTES = USED + SLACK;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(CX_BYTES + CY_BYTES == kConstBlockFloats * 4, "constant block layout");
  static_assert(OFF_CX - OFF_Q >= 16 * 4096, "epilogue staging: 4 KB per softmax warp in the Q/dO stages");
};
constexpr uint32_t KV_TM_ST = 0, KV_TM_DPT = 128, KV_TM_DV = 256, KV_TM_DK = 384;
// 16 softmax warps, four per scheduler: warp w owns TMEM lanes 32 (w % 4) .. + 31 (its key
// rows) and query columns [KV_COLS (w / 4), KV_COLS (w / 4) + KV_COLS) of every tile.
constexpr int KV_SOFTMAX_WARPS = 16;
constexpr int KV_COLS = BM * 4 / KV_SOFTMAX_WARPS;   // 32
constexpr int KV_PRODUCER_WARP = KV_SOFTMAX_WARPS;
// two MMA-issuing threads: the first issues S^T and dP^T, the second dV and dK
constexpr int KV_MMA_WARP = KV_SOFTMAX_WARPS + 1;
constexpr int KV_THREADS = 32 * (KV_SOFTMAX_WARPS + 3);
static_assert(KV_COLS == 32, "one 32-column TMEM load per softmax warp; P^T handed over in two 16-query halves");

// The masked dQ kernel runs a query tile whose row of the tile maps is a plain run of key
// tiles 0 .. n - 1 (its plain length: a key-padding mask, or an all-true one) as an unmasked one
// over the first min(N_K, 128 n) keys: its rows see exactly those keys, so the results are
// the same without the per-row mask words, the chunk votes or the tile walk.
template <int D, bool MASK>
__global__ void __launch_bounds__(DQ_THREADS, 1)
    attn_bwd_dq_tc_kernel(const AttnShape s, const __grid_constant__ BwdTcArgs args, const LaunchCtx ctx) {
  if constexpr (MASK) {
    if (args.mask_q.plain) {
      const int nqt = (s.NQ + BM - 1) / BM;
      const int item = blockIdx.x;
      const int bh = item / nqt;
      const int qt = s.causal ? (nqt - 1 - item % nqt) : (item % nqt);
      const int gm = (args.mask_q.mb > 1 ? bh / s.H : 0) * args.mask_q.mh + (args.mask_q.mh > 1 ? bh % s.H : 0);
      const int n = args.mask_q.plain[static_cast<size_t>(gm) * nqt + qt];
      if (n > 0) {
        dq_body<D, false>(s, args, ctx, min(s.NK, n * BN));
        return;
      }
    }
  }
  dq_body<D, MASK>(s, args, ctx, s.NK);
}

// MASK: a boolean attention mask (args.mask_k, rows = keys) applies on top of `causal`.
template <int D, bool MASK>
__device__ __forceinline__ void dkdv_body(const AttnShape& s, const BwdTcArgs& args, const LaunchCtx& ctx) {
  using C = DkvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t mis = smem_u32(smem_raw) & 1023u;
  if (C::SLACK == 0 && mis != 0) {   // uniform across the CTA: nothing launched yet
    if (threadIdx.x == 0) atomicOr(ctx.status, kStatusBadSmem);
    return;
  }
  uint8_t* smem = smem_raw + ((1024u - mis) & 1023u);
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sDS = smem + C::OFF_DS;
  float* st_base = reinterpret_cast<float*>(smem + C::OFF_CX);
  float* st_invs = st_base + BM;
  float* st_d = reinterpret_cast<float*>(smem + C::OFF_CY);
  float* st_r = st_d + BM;
  int* st_a = reinterpret_cast<int*>(st_d + 2 * BM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = kv_full + 1;
  uint64_t* q_empty = q_full + C::NQS;
  uint64_t* do_full = q_empty + C::NQS;
  uint64_t* do_empty = do_full + C::NDS;
  uint64_t* st_full = do_empty + C::NDS;   // S^T committed and constants X landed
  uint64_t* dpt_full = st_full + 1;   // dP^T committed and constants Y landed (after dK read dS^T)
  uint64_t* dpt_free = dpt_full + 1;
  // p_full[h]: every softmax warp has written half h of its P^T (query columns 16 h .. 16 h + 15
  // of its 32): dV takes each half as it lands
  uint64_t* p_full = dpt_free + 1;
  uint64_t* p_free = p_full + 2;
  uint64_t* acc_full = p_free + 1;
  uint64_t* drain = acc_full + 1;   // [2], one per issuer
  uint64_t* cx_empty = drain + 2;
  uint64_t* cy_empty = cx_empty + 1;
  uint64_t* ds_full = cy_empty + 1;   // dS^T tile written (P^T has p_full / p_free)
  uint64_t* ds_free = ds_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqt = (s.NQ + BM - 1) / BM;
  const int item = blockIdx.x;
  // head-major order (Q/dO of a head shared in L2); within a head ascending key tiles,
  // which under the causal mask see the most queries
  const int nkt_all = (s.NK + BN - 1) / BN;
  const int bh = item / nkt_all;
  const int kt = item % nkt_all;
  const int k0 = kt * BN;
  const int qt0 = s.causal ? k0 / BM : 0;   // first query tile that can see key k0 (j <= i)
  const int nq = max(0, nqt - qt0);
  // Query tiles 32 w .. 32 w + 31 this key tile takes, as bits (the loops run over qt0 ..
  // nqt - 1): with a tile live map, the tiles holding an allowed pair.  Every role walks
  // them in order and counts them (it): ring slots and barrier phases follow that count, so
  // a fully masked tile costs nothing.  Unmasked: every tile of the range.
  auto take_word = [&](int w) -> uint32_t {
    uint32_t bits = ~0u;
    if constexpr (MASK) {
      if (args.mask_k.live) {
        const int gm = (args.mask_k.mb > 1 ? bh / s.H : 0) * args.mask_k.mh + (args.mask_k.mh > 1 ? bh % s.H : 0);
        bits = args.mask_k.live[(static_cast<size_t>(gm) * nkt_all + kt) * args.mask_k.live_words + w];
      }
    }
    return bits;
  };
  // Query tiles 32 w .. 32 w + 31 the mask allows whole to every key of this tile: their mask
  // words are all ones and are not read.
  auto full_word = [&](int w) -> uint32_t {
    if constexpr (MASK) {
      if (args.mask_k.full) {
        const int gm = (args.mask_k.mb > 1 ? bh / s.H : 0) * args.mask_k.mh + (args.mask_k.mh > 1 ? bh % s.H : 0);
        return args.mask_k.full[(static_cast<size_t>(gm) * nkt_all + kt) * args.mask_k.live_words + w];
      }
    }
    return 0u;
  };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < C::NQS; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 2);   // S^T (issuer 0) and dK (issuer 1) read Q_i
    }
    for (int i = 0; i < C::NDS; ++i) {
      mbar_init(&do_full[i], 1);
      mbar_init(&do_empty[i], 2);   // dP^T (issuer 0) and dV (issuer 1) read dO_i
    }
    mbar_init(st_full, 2);   // issuer 0's commit + the producer's arrival for X
    mbar_init(dpt_full, 2);   // issuer 0's commit + the producer's arrival for Y
    mbar_init(dpt_free, KV_SOFTMAX_WARPS);
    // p_full[0], p_full[1] and ds_full: one counted barrier each for all query tiles.  A warp
    // that has finished tile i cannot arrive for tile i + 1 while another warp's arrival for
    // tile i is missing: its next P^T needs S^T_{i+1} (st_full), which issuer 0 issues only
    // after p_free, i.e. after the dV_i products that p_full's phases i started (the second
    // half's arrivals come after the first's in every warp); its next dS^T needs
    // Y_{i+1} (dpt_full), which the producer issues only after ds_free, i.e. after the dK_i
    // product that ds_full's phase i started.  Those two waits keep every arrival in its own
    // tile's phase; a reordering that drops either needs one barrier per buffer, as e_full in
    // the dQ kernel.
    mbar_init(&p_full[0], KV_SOFTMAX_WARPS);
    mbar_init(&p_full[1], KV_SOFTMAX_WARPS);
    mbar_init(p_free, 1);
    mbar_init(acc_full, 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(cx_empty, KV_SOFTMAX_WARPS);
    mbar_init(cy_empty, KV_SOFTMAX_WARPS);
    mbar_init(ds_full, KV_SOFTMAX_WARPS);
    mbar_init(ds_free, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == KV_MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == KV_PRODUCER_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&args.tm_q);
      tma_prefetch_desc(&args.tm_k);
      tma_prefetch_desc(&args.tm_v);
      tma_prefetch_desc(&args.tm_do);
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sK + c * BOX_BYTES, &args.tm_k, kv_full, c * 64, k0, bh);
        tma_load_3d(sV + c * BOX_BYTES, &args.tm_v, kv_full, c * 64, k0, bh);
      }
      bool ok = true;
      int q_issued = 0, d_issued = 0, cx_issued = 0, cy_issued = 0;
      uint32_t tw = ~0u;
      for (int qa = qt0, cnt = 0; qa < nqt && ok; ++qa) {
        if constexpr (MASK) {
          if (qa == qt0 || (qa & 31) == 0) tw = take_word(qa >> 5);
          if (!((tw >> (qa & 31)) & 1u)) continue;
        }
        const int it = cnt++;
        const int i0 = qa * BM;
        const int qs = it % C::NQS;
        const uint32_t cpar = (it & 1u) ^ 1u;
        const float* blk = args.ws_consts + (static_cast<size_t>(bh) * nqt + qa) * kConstBlockFloats;
        ok = mbar_wait(&q_empty[qs], ((it / C::NQS) & 1u) ^ 1u, abort_flag, ctx);
        if (!ok) break;
        mbar_arrive_expect_tx(&q_full[qs], C::TILE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sQ + qs * C::TILE + c * BOX_BYTES, &args.tm_q, &q_full[qs], c * 64, i0, bh);
        q_issued = it + 1;
        // X(it) completes on st_full phase it: the warps' arrivals on cx_empty for tile it - 1
        // come after their wait on phase it - 1
        ok = mbar_wait(cx_empty, cpar, abort_flag, ctx);
        if (!ok) break;
        mbar_arrive_expect_tx(st_full, C::CX_BYTES);
        bulk_load_1d(st_base, blk, C::CX_BYTES, st_full);
        cx_issued = it + 1;
        const int ds = it % C::NDS;
        ok = mbar_wait(&do_empty[ds], ((it / C::NDS) & 1u) ^ 1u, abort_flag, ctx);
        if (!ok) break;
        mbar_arrive_expect_tx(&do_full[ds], C::TILE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sDO + ds * C::TILE + c * BOX_BYTES, &args.tm_do, &do_full[ds], c * 64, i0, bh);
        d_issued = it + 1;
        // Y(it) completes on dpt_full phase it.  It is issued once dK of tile it - 1 has read
        // the dS^T tile, so a warp that sees dpt_full phase it may overwrite that tile.
        ok = mbar_wait(cy_empty, cpar, abort_flag, ctx) && mbar_wait(ds_free, cpar, abort_flag, ctx);
        if (!ok) break;
        mbar_arrive_expect_tx(dpt_full, C::CY_BYTES);
        bulk_load_1d(st_d, blk + 2 * BM, C::CY_BYTES, dpt_full);
        cy_issued = it + 1;
      }
      drain_wait(kv_full, 0, ctx);
      for (int it = max(0, q_issued - C::NQS); it < q_issued; ++it)
        drain_wait(&q_full[it % C::NQS], (it / C::NQS) & 1u, ctx);
      for (int it = max(0, d_issued - C::NDS); it < d_issued; ++it)
        drain_wait(&do_full[it % C::NDS], (it / C::NDS) & 1u, ctx);
      // the last X and Y copies (their phases also need the issuer's commit, which a CTA
      // winding down after a timeout may never make: the drain bound ends the wait then)
      if (cx_issued > 0) drain_wait(st_full, (cx_issued - 1) & 1u, ctx);
      if (cy_issued > 0) drain_wait(dpt_full, (cy_issued - 1) & 1u, ctx);
    }
  } else if (warp >= KV_MMA_WARP) {
    const int who = warp - KV_MMA_WARP;   // 0: S^T and dP^T products; 1: dV and dK products
    if (lane == 0) {
      constexpr uint32_t idesc_ss = idesc_fp16_f32(BN, BM, 0, 0);
      constexpr uint32_t idesc_kmn = idesc_fp16_f32(BN, D, 0, 1);
      constexpr uint32_t HI = sdesc_hi_sw128(1024);
      const uint32_t klo = sdesc_lo(smem_u32(sK), 16), vlo = sdesc_lo(smem_u32(sV), 16),
                     dslo = sdesc_lo(smem_u32(sDS), 16);
      const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO);
      bool ok = mbar_wait(kv_full, 0, abort_flag, ctx);
      // test knob: nothing is committed to `drain` yet, so this wait can only time out
      if (ok && ctx.force_timeout) ok = mbar_wait(&drain[who], 0, abort_flag, ctx);
      uint32_t tw = ~0u;
      for (int qa = qt0, cnt = 0; qa < nqt && ok; ++qa) {
        if constexpr (MASK) {
          if (qa == qt0 || (qa & 31) == 0) tw = take_word(qa >> 5);
          if (!((tw >> (qa & 31)) & 1u)) continue;
        }
        const int it = cnt++;
        const int qs = it % C::NQS, ds = it % C::NDS;
        const uint32_t par = it & 1u;
        if (who == 0) {
          // S^T = K Q_i^T
          ok = mbar_wait(&q_full[qs], (it / C::NQS) & 1u, abort_flag, ctx) &&
               mbar_wait(p_free, par ^ 1u, abort_flag, ctx);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qlo = sdesc_lo(aQ + qs * C::TILE, 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
            tc_mma_f16(tmem + KV_TM_ST, sdesc(klo + off, HI), sdesc(qlo + off, HI), idesc_ss, kk > 0 ? 1u : 0u);
          }
          tc_commit(st_full);
          tc_commit(&q_empty[qs]);
          // dP^T = V dO_i^T
          ok = mbar_wait(&do_full[ds], (it / C::NDS) & 1u, abort_flag, ctx) &&
               mbar_wait(dpt_free, par ^ 1u, abort_flag, ctx);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dolo = sdesc_lo(aDO + ds * C::TILE, 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
            tc_mma_f16(tmem + KV_TM_DPT, sdesc(vlo + off, HI), sdesc(dolo + off, HI), idesc_ss, kk > 0 ? 1u : 0u);
          }
          tc_commit(dpt_full);
          tc_commit(&do_empty[ds]);
        } else {
          // dV += P^T dO_i as soon as P^T is written (its release lets S^T of the next
          // tile be issued and the producer load the next dO), then dK += dS^T Q_i.
          // Q_i and dO_i arrived long before: waiting on them first leaves a single wait
          // between the softmax warps' arrival and the first product.
          ok = mbar_wait(&q_full[qs], (it / C::NQS) & 1u, abort_flag, ctx) &&
               mbar_wait(&do_full[ds], (it / C::NDS) & 1u, abort_flag, ctx);
          if (!ok) break;
          const uint32_t qmn = sdesc_lo(aQ + qs * C::TILE, BOX_BYTES), domn = sdesc_lo(aDO + ds * C::TILE, BOX_BYTES);
          // two halves: the first 16 query columns of every softmax warp (16-query steps kk =
          // 0, 2, 4, 6), issued while the warps form the second 16 (kk = 1, 3, 5, 7)
          for (int h = 0; h < 2 && ok; ++h) {
            ok = mbar_wait(&p_full[h], par, abort_flag, ctx);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kq = 0; kq < BM / 32; ++kq) {
              const int kk = 2 * kq + h;
              // P^T from tensor memory: the softmax warps of queries 16 kk .. 16 kk + 15 wrote
              // it over the first half of their S^T columns, 8 columns per 16 queries
              tc_mma_f16_ts(tmem + KV_TM_DV,
                            tmem + KV_TM_ST + (16 * kk / KV_COLS) * KV_COLS + (16 * kk % KV_COLS) / 2,
                            sdesc(domn + ((kk * 2048) >> 4), HI), idesc_kmn, (it > 0 || kk > 0) ? 1u : 0u);
            }
          }
          if (!ok) break;
          tc_commit(&do_empty[ds]);
          tc_commit(p_free);
          ok = mbar_wait(ds_full, par, abort_flag, ctx);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) {
            const uint32_t aoff = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
            tc_mma_f16(tmem + KV_TM_DK, sdesc(dslo + aoff, HI), sdesc(qmn + ((kk * 2048) >> 4), HI), idesc_kmn,
                       (it > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&q_empty[qs]);
          tc_commit(ds_free);
        }
      }
      if (ok && who == 1) tc_commit(acc_full);
      tc_commit(&drain[who]);
      drain_wait(&drain[who], 0, ctx);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps (row = key)
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31 (key rows) and query columns
    // [64 (w / 4), 64 (w / 4) + 64) of every tile.
    const int quarter = warp & 3;
    const int part = warp >> 2;
    const int cbase = part * KV_COLS;
    const int r = quarter * 32 + lane;
    const int j = k0 + r;
    const bool j_ok = j < s.NK;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = s.scale * (1.0f / 32.0f);
    bool ok = true;
    // A wait that gives up sets ok = false; the loop still runs to the end without
    // waiting (its named barriers must be reached by all eight warps) and the
    // epilogue is skipped.
    auto warp_wait = [&](uint64_t* bar, uint32_t par) {
      if (!ok) return;
      int okv = 1;
      if (lane == 0) okv = mbar_wait(bar, par, abort_flag, ctx) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, okv, 0) != 0;
    };
    // this key row's attention-mask words (the transposed mask): four per query tile
    const uint32_t* mkey = nullptr;
    if (MASK) {
      const int gm = (args.mask_k.mb > 1 ? bh / s.H : 0) * args.mask_k.mh + (args.mask_k.mh > 1 ? bh % s.H : 0);
      mkey = args.mask_k.bits + (static_cast<size_t>(gm) * s.NK + (j_ok ? j : s.NK - 1)) * args.mask_k.words;
    }
    uint32_t sv[KV_COLS / 32][32];
#define SV(c) sv[(c) >> 5][(c) & 31]
    uint32_t tw = ~0u, fw = 0;
    int ntaken = 0;   // query tiles taken; 0 leaves the dK and dV accumulators unwritten
    for (int qa = qt0; qa < nqt; ++qa) {
      if constexpr (MASK) {
        if (qa == qt0 || (qa & 31) == 0) {
          tw = take_word(qa >> 5);
          fw = full_word(qa >> 5);
        }
        if (!((tw >> (qa & 31)) & 1u)) continue;
      }
      const int it = ntaken++;
      const int i0 = qa * BM;
      const uint32_t par = it & 1u;
      // S^T and this tile's per-query constants X (queries past N_Q carry base 2: zero weight)
      // in flight during the wait; a tile the mask allows whole reads none
      const uint32_t mw = (MASK && !((fw >> (qa & 31)) & 1u)) ? mkey[4 * qa + part] : ~0u;
      warp_wait(st_full, par);
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < KV_COLS / 32; ++h) tmem_ld32(lane_addr + KV_TM_ST + cbase + 32 * h, sv[h]);
      tc_wait_ld();
      // masked: key past N_K, or (causal) query i0 + c < j
      const int first_vis = !j_ok ? BM : (s.causal ? min(BM, max(0, j - i0)) : 0);   // first visible column
      // With an attention mask, a chunk every key row of the warp sees whole needs no per-entry
      // test, and a chunk none of them sees has zero P^T and dS^T (no constants read, no
      // arithmetic).  The vote runs in the masked instance only, where the whole warp is here
      // together.
      int kind = kChunkMixed;
      if constexpr (MASK) kind = chunk_vote(mw == ~0u && first_vis <= cbase, mw == 0u || first_vis >= cbase + KV_COLS);
      const bool need_mask = MASK ? kind == kChunkMixed : (!j_ok || (s.causal && i0 + cbase < j));
      const bool dead = MASK && kind == kChunkNone;
      // P^T = q^8 / s_i and the dS coefficient q^7 (1/w)^2 / s_i = q^7 (1 + q)^2 / s_i (in
      // place): with t = q^7 / s_i, P = t q and the coefficient is t + P (2 + q).  The factor
      // 1/4 comes with dP^T - D_i below.  Four entries share two reciprocals (as in coef_quad).
      // P^T goes to tensor memory as fp16 pairs over the first half of this warp's S^T
      // columns (already read; S^T of the next tile is issued only after dV has read P^T).
      uint32_t pt[16];
#pragma unroll
      for (int c = 0; c < KV_COLS; c += 8) {
        uint32_t* pk = pt + ((c & 31) >> 1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cb = c + 4 * h;        // local column
          const int cg = cbase + cb;       // column in the tile
          if (dead) {
            SV(cb) = SV(cb + 1) = SV(cb + 2) = SV(cb + 3) = 0u;
            pk[2 * h] = pk[2 * h + 1] = 0u;
            continue;
          }
          const float4 b4 = *reinterpret_cast<const float4*>(st_base + cg);
          const float4 i4 = *reinterpret_cast<const float4*>(st_invs + cg);
          float x[4] = {u2f(SV(cb)), u2f(SV(cb + 1)), u2f(SV(cb + 2)), u2f(SV(cb + 3))};
          if (need_mask) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (cg + t < first_vis || (MASK && !((mw >> (cb + t)) & 1u))) x[t] = -INFINITY;
          }
          const float2 A = make_float2(fma_sat(x[0], -c2, b4.x), fma_sat(x[1], -c2, b4.y));
          const float2 B = make_float2(fma_sat(x[2], -c2, b4.z), fma_sat(x[3], -c2, b4.w));
          const float2 PR = __fmul2_rn(A, B);
          const float2 R = make_float2(rcp_approx(PR.x), rcp_approx(PR.y));
          const float2 m1 = make_float2(-1.0f, -1.0f), two = make_float2(2.0f, 2.0f);
          const float2 qa = __ffma2_rn(R, B, m1), qb = __ffma2_rn(R, A, m1);   // 1/w - 1
          const float2 qa2 = __fmul2_rn(qa, qa), qb2 = __fmul2_rn(qb, qb);
          const float2 qa7 = __fmul2_rn(__fmul2_rn(qa2, qa2), __fmul2_rn(qa2, qa));
          const float2 qb7 = __fmul2_rn(__fmul2_rn(qb2, qb2), __fmul2_rn(qb2, qb));
          const float2 ta = __fmul2_rn(qa7, make_float2(i4.x, i4.y)), tb = __fmul2_rn(qb7, make_float2(i4.z, i4.w));
          const float2 pa = __fmul2_rn(ta, qa), pb = __fmul2_rn(tb, qb);
          const float2 ca = __ffma2_rn(pa, __fadd2_rn(qa, two), ta);
          const float2 cbv = __ffma2_rn(pb, __fadd2_rn(qb, two), tb);
          SV(cb) = __float_as_uint(ca.x);
          SV(cb + 1) = __float_as_uint(ca.y);
          SV(cb + 2) = __float_as_uint(cbv.x);
          SV(cb + 3) = __float_as_uint(cbv.y);
          pk[2 * h] = pack_f16x2_sat(pa.x, pa.y);
          pk[2 * h + 1] = pack_f16x2_sat(pb.x, pb.y);
        }
        if (c == 8) {   // the first 16 queries' P^T: dV starts on it while the rest is formed
          tmem_st8(lane_addr + KV_TM_ST + cbase, pt);
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[0]);
        }
      }
      tmem_st8(lane_addr + KV_TM_ST + cbase + 8, pt + 8);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(cx_empty);   // this warp's reads of X are done
        mbar_arrive(&p_full[1]);
      }
      // dS^T = coef (dP^T - D_i); the entries (a_i, i) where this key is the query's argmax
      // take -R_i afterwards
      // dP^T, the constants Y, and (through the producer) dK of the previous tile done
      warp_wait(dpt_full, par);
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < KV_COLS / 32; ++cc) {
        uint32_t dv[32];
        tmem_ld32(lane_addr + KV_TM_DPT + cbase + cc * 32, dv);
        tc_wait_ld();
        if (cc == KV_COLS / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dpt_free);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int cb = cc * 32 + e * 8;
          const int cg = cbase + cb;
          uint32_t pk[4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (dead) {
              pk[2 * h] = pk[2 * h + 1] = 0u;
              continue;
            }
            const float4 d4 = *reinterpret_cast<const float4*>(st_d + cg + 4 * h);   // D_i / 4
            const int c = cb + 4 * h;
            const float2 q4 = make_float2(0.25f, 0.25f);
            // coef (dP - D_i) / 4 = coef (dP / 4 - D_i / 4)
            const float2 v0 = __fmul2_rn(make_float2(u2f(SV(c)), u2f(SV(c + 1))),
                                         __ffma2_rn(make_float2(u2f(dv[e * 8 + 4 * h]), u2f(dv[e * 8 + 4 * h + 1])), q4,
                                                    make_float2(-d4.x, -d4.y)));
            const float2 v1 = __fmul2_rn(make_float2(u2f(SV(c + 2)), u2f(SV(c + 3))),
                                         __ffma2_rn(make_float2(u2f(dv[e * 8 + 4 * h + 2]), u2f(dv[e * 8 + 4 * h + 3])), q4,
                                                    make_float2(-d4.z, -d4.w)));
            pk[2 * h] = pack_f16x2_sat(v0.x, v0.y);
            pk[2 * h + 1] = pack_f16x2_sat(v1.x, v1.y);
          }
          st_tile16(sDS, r, cg >> 3, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        }
      }
      // Argmax entries in this warp's rows and columns: -R_i replaces the value at
      // (a_i - k0, i).  Lane l looks at columns cbase + l (+ 32 ...); about
      // BN / N_K of a tile's queries have their argmax among this CTA's keys.
      __syncwarp();   // the row owners' stores above come first
#pragma unroll
      for (int wd = 0; wd < KV_COLS / 32; ++wd) {
        const int col = cbase + 32 * wd + lane;
        const int rr = st_a[col] - k0;
        if (rr >= quarter * 32 && rr < quarter * 32 + 32) {
          const int chunk = col >> 3;
          const uint32_t h16 = pack_f16x2_sat(-st_r[col], 0.0f) & 0xffffu;
          *reinterpret_cast<unsigned short*>(sDS + (chunk >> 3) * BOX_BYTES + rr * 128 +
                                             (((chunk & 7) ^ (rr & 7)) << 4) + (col & 7) * 2) =
              static_cast<unsigned short>(h16);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(cy_empty);   // this warp's reads of Y are done
        mbar_arrive(ds_full);
      }
    }
#undef SV
    if (ntaken > 0) warp_wait(acc_full, 0);
    if (ok) {
      tc_fence_after();
      // the warps of a row quarter store 32-column chunks of its key rows in turn, through
      // 4 KB per warp of the Q/dO stages (free: acc_full means every product has completed)
      uint8_t* stage = sQ + warp * 4096;
      const int wrow0 = k0 + quarter * 32;   // first key row of this warp
      const size_t row0 = static_cast<size_t>(bh) * s.NK + wrow0;
      const int n_ok = max(0, min(32, s.NK - wrow0));
#pragma unroll
      for (int c0 = part * 32; c0 < D; c0 += 32 * (KV_SOFTMAX_WARPS / 4)) {
        uint32_t av[32], kv[32];
        tmem_ld32(lane_addr + KV_TM_DV + c0, av);
        tmem_ld32(lane_addr + KV_TM_DK + c0, kv);
        tc_wait_ld();
        float ov[32], okv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          ov[e] = ntaken > 0 ? u2f(av[e]) : 0.0f;
          okv[e] = ntaken > 0 ? s.scale * u2f(kv[e]) : 0.0f;
        }
        if (args.grad_bf16) {
          warp_store_block32<true>(stage, ov, args.dv, row0, D, c0, n_ok, lane);
          warp_store_block32<true>(stage, okv, args.dk, row0, D, c0, n_ok, lane);
        } else {
          warp_store_block32<false>(stage, ov, args.dv, row0, D, c0, n_ok, lane);
          warp_store_block32<false>(stage, okv, args.dk, row0, D, c0, n_ok, lane);
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == KV_MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// The masked dK/dV kernel runs a key tile whose every query tile in range the mask allows
// whole (its plain flag: its row of the full map covers the range) as an unmasked one: the
// same results without the per-key mask words, the chunk votes or the tile walk.
template <int D, bool MASK>
__global__ void __launch_bounds__(KV_THREADS, 1)
    attn_bwd_dkdv_tc_kernel(const AttnShape s, const __grid_constant__ BwdTcArgs args, const LaunchCtx ctx) {
  if constexpr (MASK) {
    if (args.mask_k.plain) {
      const int nkt_all = (s.NK + BN - 1) / BN;
      const int item = blockIdx.x;
      const int bh = item / nkt_all;
      const int kt = item % nkt_all;
      const int gm = (args.mask_k.mb > 1 ? bh / s.H : 0) * args.mask_k.mh + (args.mask_k.mh > 1 ? bh % s.H : 0);
      const bool whole = args.mask_k.plain[static_cast<size_t>(gm) * nkt_all + kt] != 0;
      if (whole) {
        dkdv_body<D, false>(s, args, ctx);
        return;
      }
    }
  }
  dkdv_body<D, MASK>(s, args, ctx);
}

template <typename KernelFn>
cudaError_t set_smem(KernelFn fn, int bytes) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, bool MASK>
cudaError_t launch_bwd_d(const AttnShape& s, const BwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st,
                         const KernelEvents& ev) {
  cudaError_t e = set_smem(attn_bwd_dq_tc_kernel<D, MASK>, DqCfg<D>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = set_smem(attn_bwd_dkdv_tc_kernel<D, MASK>, DkvCfg<D>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned BH = static_cast<unsigned>(s.B * s.H);
  const unsigned nqt = static_cast<unsigned>((s.NQ + BM - 1) / BM);
  const unsigned nkt = static_cast<unsigned>((s.NK + BN - 1) / BN);
  ConvertJob job;
  const size_t nq8 = static_cast<size_t>(BH) * s.NQ * D / 8, nk8 = static_cast<size_t>(BH) * s.NK * D / 8;
  const void* srcs[4] = {a.q_raw, a.k_raw, a.v_raw, a.dout};
  void* dsts[4] = {a.q16, a.k16, a.v16, a.do16};
  const size_t ns[4] = {nq8, nk8, nk8, nq8};
  for (int i = 0; i < 4; ++i) {
    job.src[i] = static_cast<const uint4*>(srcs[i]);
    job.dst[i] = static_cast<uint4*>(dsts[i]);
    job.n8[i] = ns[i];
  }
  job.count = 4;
  if ((e = ev.rec(0, st)) != cudaSuccess) return e;
  e = launch_bf16_to_f16(job, ctx.status, st);
  if (e != cudaSuccess) return e;
  if ((e = ev.rec(1, st)) != cudaSuccess) return e;
  attn_bwd_dq_tc_kernel<D, MASK><<<nqt * BH, DQ_THREADS, DqCfg<D>::SMEM_BYTES, st>>>(s, a, ctx);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = ev.rec(2, st)) != cudaSuccess) return e;
  attn_bwd_dkdv_tc_kernel<D, MASK><<<nkt * BH, KV_THREADS, DkvCfg<D>::SMEM_BYTES, st>>>(s, a, ctx);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return ev.rec(3, st);
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const AttnShape& s, const BwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st,
                               const KernelEvents& ev) {
  const bool mask = a.mask_q.bits != nullptr;
  if (s.D == 128)
    return mask ? launch_bwd_d<128, true>(s, a, ctx, st, ev) : launch_bwd_d<128, false>(s, a, ctx, st, ev);
  if (s.D == 64)
    return mask ? launch_bwd_d<64, true>(s, a, ctx, st, ev) : launch_bwd_d<64, false>(s, a, ctx, st, ev);
  return cudaErrorInvalidValue;
}

}  // namespace raattn
