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
// One CTA owns TWO 128-row query tiles (A: rows q0 .. q0+127, B: q0+128 .. q0+255) of
// one (batch, head) and runs both passes over the key tiles they can see.  Every K and
// V tile brought into shared memory serves both query tiles: the tile loads into one
// SM top out near 40-46 bytes per clock, and one query tile per CTA would need about
// 62 bytes per clock to keep the tensor core busy (K twice and V once per 1536
// tensor cycles at D = 128); two query tiles halve that.
//   warp 8      TMA producer: Q_A and Q_B once, then K tiles (pass 1), then K and V
//               tiles interleaved in the order the MMA thread consumes them (pass 2),
//               through a ring of NSTAGE shared-memory stages.
//   warps 9, 10 MMA issuers, one thread per query tile g: S_g = Q_g K^T into its TMEM
//               score buffer (128 x 128 fp32); in pass 2 also O_g += P_g V into its TMEM
//               accumulator (128 x D fp32), issued as S_g(j+1) then O_g(j) so the softmax
//               warpgroup works on S_g(j+1) while O_g(j) runs.  Each issuer waits on its
//               own barriers; a wait stalls the issuing thread for a few hundred cycles,
//               longer than the two 64-cycle products the tensor queue holds, and with two
//               issuers the other tile's products keep the tensor core busy meanwhile.
//   warps 0-3   softmax warpgroup of query tile A, warps 4-7 that of tile B; thread t of
//               a warpgroup owns query row t (TMEM lane t) and all 128 key columns:
//               pass 1 keeps the running max of the raw scores and the 32-column chunk
//               of its first occurrence, pass 2 the lowest column holding it there;
//               pass 2 forms phi on the FMA pipe (no exp), writes P = fp16(phi) into
//               its 128-byte-swizzled shared-memory tile, sums phi in fp32, and votes
//               whether the tile is live.  Epilogue: O = acc / sum(phi) and the row
//               statistics for the backward.
//   V arrives as the fp16 copy the C-ABI layer made once per call (exact for bf16
//   values from 2^-14 to 65504), so the P V product runs in fp16 and P is rounded to 2^-11
//   rather than 2^-8.  Q K^T stays in bf16.
//
// CTA pairs (D = 128, N_Q > 256): a cluster of two CTAs runs the same roles on four query
// tiles.  Product g is one M = 256 tcgen05.mma (cta_group::2) issued by the even CTA's
// issuer g: its rows 0..127 are the even CTA's tile g, rows 128..255 the odd CTA's, and
// each CTA holds only its half of every K tile (64 keys) and V tile (64 columns).  Both
// CTAs' copies complete on the even CTA's ring and Q barriers (the even producer arms them
// for both); the issuer's commits land on both CTAs' barriers; the odd CTA's softmax warps
// arrive on the even CTA's score-free and P-full barriers; the pair meets at a cluster
// barrier after set-up and before the tensor memory is freed.
//
// phi on the FMA pipe: w = (1+u)/2 = 0.5 + (m - s)/32 (scaled units) computed with
// one saturating FMA, so every u >= 1 (and every masked entry, fed as -inf) gives
// w = 1; q = 1/w - 1; phi = ((q^2)^2)^2.  Four scores share two reciprocals: with the
// pairs A = (w0, w1), B = (w2, w3), R = 1/(A B) elementwise gives R B = (1/w0, 1/w1)
// and R A = (1/w2, 1/w3), halving the special-function-unit work, and the rest runs
// as packed f32x2 operations.  At w = 1 the computed q is below 3e-7, so phi rounds to
// exactly 0.0.
#include "kernels.cuh"
#include "phi.cuh"

namespace raattn {
namespace {

constexpr int BM = 128;   // query rows per tile: the MMA M and the 128 TMEM lanes
constexpr int BN = 128;   // keys per tile: the N of Q K^T and the K of P V
constexpr int NGROUP = 2;                            // query tiles per CTA
constexpr int GROUP_WARPS = 4;                       // one warpgroup per query tile
constexpr int SOFTMAX_WARPS = NGROUP * GROUP_WARPS;  // 8
constexpr int PRODUCER_WARP = SOFTMAX_WARPS;
constexpr int MMA_WARP = SOFTMAX_WARPS + 1;          // MMA_WARP + g issues the products of query tile g
constexpr int THREADS = 32 * (SOFTMAX_WARPS + 1 + NGROUP);
constexpr int CAUSAL_HEADS = 64;  // causal CTA order: heads per longest-first group
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S = 0;     // S of query tile g at column 128 g
constexpr uint32_t TMEM_O = 256;   // O of query tile g at column 256 + 128 g
constexpr int BOX_BYTES = 128 * 64 * 2;   // one TMA box: 128 rows x 64 16-bit values (128 B per row)
constexpr int HALF_BOX_BYTES = 64 * 64 * 2;   // 64 rows x 64 values: a pair CTA's share of a K box

// PAIR: the kernel runs as a cluster of two CTAs on the two SMs of a TPC.  Each product
// is one M = 256 tcgen05.mma (cta_group::2) issued by the even CTA: query rows 0..127 of
// it are the even CTA's tile g, rows 128..255 the odd CTA's, and each CTA holds only half
// of every K tile (64 keys) and of every V tile (64 of the D columns).  Per SM that halves
// the K/V copies and the shared-memory reads of the B operands, the limit of the
// single-CTA form.
template <int D, bool PAIR>
struct FwdCfg {
  static constexpr int NCTA = PAIR ? 2 : 1;
  static constexpr int TILE_BYTES = BN * D * 2;   // a Q, K or V tile: D/64 boxes
  static constexpr int STAGE_BYTES = TILE_BYTES / NCTA;   // this CTA's part of a K or V tile
  // Ring depth: K/V tiles in flight; each stage serves two products (S_A and S_B, or
  // O_A and O_B).
  static constexpr int NSTAGE = NCTA * ((D == 128) ? 3 : 6);
  static constexpr int P_BYTES = BM * BN * 2;     // P tile: two 64-key halves of 16 KB
  static constexpr int OFF_Q = 0;                 // Q_A, Q_B
  static constexpr int OFF_RING = OFF_Q + NGROUP * TILE_BYTES;
  static constexpr int OFF_P = OFF_RING + NSTAGE * STAGE_BYTES;   // P_A, P_B
  static constexpr int OFF_BAR = OFF_P + NGROUP * P_BYTES;
  // q_full, ring_full[NSTAGE], ring_empty[NSTAGE], s_full[2][2], s_empty[2][2], p_full[2], p_empty[2],
  // o_full[2], drain[2]
  static constexpr int NUM_BARS = 1 + 2 * NSTAGE + 8 * NGROUP;
  static constexpr int OFF_MISC = (OFF_BAR + NUM_BARS * 8 + 15) / 16 * 16;
  // tmem base, abort flag, the odd CTA producer's fill count (pair), pad; live votes (16-byte aligned)
  static constexpr int MISC_BYTES = 16 + SOFTMAX_WARPS * 4;
  static constexpr int USED = OFF_MISC + MISC_BYTES;
  // alignment slack only where it fits; otherwise the kernel requires (and checks) a
  // 1024-byte aligned dynamic shared-memory base
  static constexpr int SLACK = (USED + 1024 <= 232448) ? 1024 : 0;
  static constexpr int SMEM_BYTES = USED + SLACK;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Pass-2 arithmetic of one 64-key half of a row, held in h (two 32-column chunks): phi
// as packed fp16 pairs in pk (four per 16-byte chunk of P) and the partial row sum.
// MASKED: columns past `lim` (causal diagonal, ragged tail) get s = -inf, hence w = 1
// and phi = 0.  BITS: so do columns whose attention-mask bit (mw0 for the first 32
// columns, mw1 for the second) is clear.
template <bool MASKED, bool BITS>
__device__ __forceinline__ float2 phi_half(const uint32_t (&h)[2][32], uint32_t (&pk)[32], int col0, int lim,
                                           float c2, float base, uint32_t mw0, uint32_t mw1) {
  float2 tsum2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = c8 * 8 + e;
      x[e] = u2f(h[c >> 5][c & 31]);
      if (MASKED && col0 + c > lim) x[e] = -INFINITY;
      if (BITS && !((((c >> 5) ? mw1 : mw0) >> (c & 31)) & 1u)) x[e] = -INFINITY;
    }
    float2 p0, p1, p2, p3;
    phi_quad(x[0], x[1], x[2], x[3], c2, base, p0, p1);
    phi_quad(x[4], x[5], x[6], x[7], c2, base, p2, p3);
    tsum2 = __fadd2_rn(tsum2, __fadd2_rn(__fadd2_rn(p0, p1), __fadd2_rn(p2, p3)));
    pk[4 * c8 + 0] = pack_f16x2_sat(p0.x, p0.y);
    pk[4 * c8 + 1] = pack_f16x2_sat(p1.x, p1.y);
    pk[4 * c8 + 2] = pack_f16x2_sat(p2.x, p2.y);
    pk[4 * c8 + 3] = pack_f16x2_sat(p3.x, p3.y);
  }
  return tsum2;
}

// One 64-key half of a P row (128 bytes) into its half of the 128-byte-swizzled tile:
// 16-byte chunk c lands at position c xor (row mod 8).
__device__ __forceinline__ void store_p_half(const uint32_t (&pk)[32], uint8_t* phalf_row, int row_local) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(phalf_row + ((c ^ (row_local & 7)) << 4)) =
        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}

// phi of one 64-key half (phi_half) through the cheapest path the warp's rows allow: with an
// attention mask, a half every row sees whole runs unmasked, a half no row sees gives zeros
// without the arithmetic, anything else the per-entry masked path; without one, the causal
// `masked` flag decides as before.
// With MASK it votes over the warp (chunk_kind): called by all lanes together.
template <bool MASK>
__device__ __forceinline__ float2 phi_half_any(bool masked, const uint32_t (&h)[2][32], uint32_t (&pk)[32], int col0,
                                               int lim, float c2, float base, uint32_t mw0, uint32_t mw1) {
  if constexpr (MASK) {
    const int k0 = chunk_kind(mw0, col0, lim), k1 = chunk_kind(mw1, col0 + 32, lim);
    if (k0 == kChunkNone && k1 == kChunkNone) {
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = 0u;
      return make_float2(0.0f, 0.0f);
    }
    if (k0 == kChunkAll && k1 == kChunkAll) return phi_half<false, false>(h, pk, col0, lim, c2, base, ~0u, ~0u);
    return phi_half<true, true>(h, pk, col0, lim, c2, base, mw0, mw1);
  } else {
    return masked ? phi_half<true, false>(h, pk, col0, lim, c2, base, ~0u, ~0u)
                  : phi_half<false, false>(h, pk, col0, lim, c2, base, ~0u, ~0u);
  }
}

// The work item of this CTA (pair): its (batch, head) bh and first query row q0; the item
// spans NCTA * NGROUP query tiles.
// Head-major order: the ~150 resident CTAs share a few heads, so each head's K and V
// stay in L2 across its query tiles.  Causal: CTA lengths differ, so heads are taken in
// groups of CAUSAL_HEADS and within a group the longest CTAs of all its heads go first;
// only the last group's short CTAs are left for the tail.  With 64 heads per group the
// resident CTAs still come two or three to a head, of nearly equal length, so they walk
// that head's keys together and L2 serves the repeated reads.
template <bool PAIR>
__device__ __forceinline__ void fwd_item(const AttnShape& s, int& bh, int& q0) {
  constexpr int NCTA = PAIR ? 2 : 1;
  const int nqt = (s.NQ + BM - 1) / BM;
  const int nct = (nqt + NCTA * NGROUP - 1) / (NCTA * NGROUP);   // work items (CTAs or pairs) per (batch, head)
  const int item = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  int ct;
  if (s.causal) {
    const int grp = item / (CAUSAL_HEADS * nct);
    const int gsize = min(CAUSAL_HEADS, s.B * s.H - grp * CAUSAL_HEADS);
    const int i = item - grp * CAUSAL_HEADS * nct;
    ct = nct - 1 - i / gsize;
    bh = grp * CAUSAL_HEADS + i % gsize;
  } else {
    bh = item / nct;
    ct = item % nct;
  }
  q0 = ct * (NCTA * NGROUP * BM);
}

// Masked calls: the number of leading keys nk > 0 over which an item may run as an unmasked
// one, or 0.  It may when every query tile of it (below N_Q) has the same plain length n > 0
// (the mask's rows of the tile maps are key tiles 0 .. n - 1, the same in both: a key-padding
// mask, or an all-true one): each of its rows then may see exactly the keys before
// nk = min(N_K, 128 n) (and the causal limit), as in an unmasked call on those keys alone, and
// the unmasked code gives the same results without the per-row mask words, the chunk votes
// or the tile walk.  Every thread of both CTAs of a pair reads the same lengths and takes the
// same decision.
template <bool PAIR>
__device__ __forceinline__ int fwd_plain_keys(const AttnShape& s, const FwdTcArgs& args, int bh, int q0) {
  constexpr int NT = (PAIR ? 2 : 1) * NGROUP;   // query tiles of the item
  if (!args.mask.plain) return 0;
  const int nqt = (s.NQ + BM - 1) / BM;
  const int gm = (args.mask.mb > 1 ? bh / s.H : 0) * args.mask.mh + (args.mask.mh > 1 ? bh % s.H : 0);
  const int* len = args.mask.plain + static_cast<size_t>(gm) * nqt;
  int n[NT];
#pragma unroll
  for (int r = 0; r < NT; ++r) n[r] = q0 / BM + r < nqt ? len[q0 / BM + r] : -1;   // -1: past N_Q
  bool same = n[0] > 0;
#pragma unroll
  for (int r = 1; r < NT; ++r) same = same && (n[r] < 0 || n[r] == n[0]);
  return same ? min(s.NK, n[0] * BN) : 0;
}

// MASK: a boolean attention mask (args.mask) applies on top of `causal`.  PAIR: the CTA
// pair form (FwdCfg).  nk: the keys taken, N_K, or fewer for an item run as an unmasked one
// over the keys its mask leaves (fwd_plain_keys).
template <int D, bool MASK, bool PAIR>
__device__ __forceinline__ void fwd_body(const AttnShape& s, const FwdTcArgs& args, const LaunchCtx& ctx, int nk) {
  using C = FwdCfg<D, PAIR>;
  constexpr int NST = C::NSTAGE;
  constexpr int NCTA = C::NCTA;
  // a pair CTA holds V columns rank * 64 .. + 63: one 128-byte swizzle atom; and no early
  // return may leave the other CTA of the pair waiting
  static_assert(!PAIR || (D == 128 && C::SLACK != 0), "CTA pair form: D = 128 with alignment slack");
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
  uint64_t* s_full = ring_empty + NST;     // [NGROUP][2]: score buffer b of query tile g at 2 g + b
  uint64_t* s_empty = s_full + 2 * NGROUP;
  uint64_t* p_full = s_empty + 2 * NGROUP;
  uint64_t* p_empty = p_full + NGROUP;
  uint64_t* o_full = p_empty + NGROUP;   // [NGROUP]
  uint64_t* drain = o_full + NGROUP;     // [NGROUP]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  // pair: ring fills the odd CTA's producer issued, stored into the even CTA's slot
  volatile uint32_t* odd_fills = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 8);
  // [NGROUP][GROUP_WARPS] votes of this CTA's softmax warps: whether the last P tile has a
  // nonzero entry, tagged with its key tile (2 j + live)
  volatile int* live = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // CTA of the pair; 0 issues the products
  const int nqt = (s.NQ + BM - 1) / BM;
  int bh, q0;
  fwd_item<PAIR>(s, bh, q0);
  // first row of query tile g of CTA r: product g spans rows q0 + NCTA BM g .. + NCTA BM - 1,
  // the even CTA's tile first
  auto tile_row0 = [&](int g, int r) { return q0 + (g * NCTA + r) * BM; };
  // last key any row of the CTA (pair) may see, and per query tile
  auto last_key_of = [&](int rows_end) {   // rows_end: one past the last row of the range
    return s.causal ? min(nk - 1, min(s.NQ - 1, rows_end - 1)) : nk - 1;
  };
  const int nkt = last_key_of(q0 + NCTA * NGROUP * BM) / BN + 1;
  // key tiles product g needs (causal: fewer for g = 0, whose rows end earlier); the
  // producer streams all nkt for the last product, and the other issuer releases the
  // stages it does not use
  auto group_keys = [&](int g) { return last_key_of(tile_row0(g, NCTA - 1) + BM) / BN + 1; };
  // Key tiles 32 w .. 32 w + 31 that product g takes, as bits: its causal range and, with a
  // tile live map, the tiles holding an allowed pair for one of its query tiles.  Every role
  // walks the same tiles in key order, refreshing its word every 32: the producer streams
  // those either product takes (a tile neither takes is left out of both passes: no copy, no
  // product, no softmax work); each issuer issues only its own product's and waits on and
  // releases the others.  Unmasked instances take the whole range.
  auto take_word = [&](int g, int w) -> uint32_t {
    const int n = group_keys(g) - 32 * w;
    uint32_t bits = n >= 32 ? ~0u : (n > 0 ? (1u << n) - 1u : 0u);
    if constexpr (MASK) {
      if (args.mask.live && bits) {
        const int gm = (args.mask.mb > 1 ? bh / s.H : 0) * args.mask.mh + (args.mask.mh > 1 ? bh % s.H : 0);
        uint32_t any = 0;
#pragma unroll
        for (int r = 0; r < NCTA; ++r) {
          const int qt = tile_row0(g, r) / BM;
          if (qt < nqt) any |= args.mask.live[(static_cast<size_t>(gm) * nqt + qt) * args.mask.live_words + w];
        }
        bits &= any;
      }
    }
    return bits;
  };
  auto union_word = [&](int w) {
    uint32_t u = 0;
#pragma unroll
    for (int h = 0; h < NGROUP; ++h) u |= take_word(h, w);
    return u;
  };
  auto bit = [](uint32_t word, int j) { return ((word >> (j & 31)) & 1u) != 0u; };
  // Barrier operations of the pair form: arrivals go to the even CTA's barrier, products and
  // commits span both CTAs.  Arrivals release, and waits acquire, at CTA scope: what they
  // order is this SM's own shared and tensor memory (a P tile, the scores a warp has read)
  // against the pair's tensor-core work, not data that the other CTA's threads read.  A
  // cluster-scope release costs about a thousand cycles per arrival (measured), on the
  // critical path of every key tile.  The one value read across the pair by threads, the
  // odd CTA's live votes, is tagged with its key tile and read after the p_full wait, so a
  // vote that is not yet visible only makes the product run.
  auto wait_bar = [&](uint64_t* bar, uint32_t par) { return mbar_wait(bar, par, abort_flag, ctx); };
  auto arrive_even = [&](uint64_t* bar) {
    if constexpr (PAIR) mbar_arrive_remote(mapa_shared(smem_u32(bar), 0));
    else mbar_arrive(bar);
  };
  auto commit = [&](uint64_t* bar) {
    if constexpr (PAIR) tc_commit_pair(bar);
    else tc_commit(bar);
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], NGROUP);   // one commit per issuer
    }
    for (int g = 0; g < NGROUP; ++g) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&s_full[2 * g + b], 1);
        mbar_init(&s_empty[2 * g + b], NCTA * GROUP_WARPS);   // one arrival per warp of the group(s)
      }
      mbar_init(&p_full[g], NCTA * GROUP_WARPS);
      mbar_init(&p_empty[g], 1);
      mbar_init(&o_full[g], 1);
      mbar_init(&drain[g], 1);
    }
    *abort_flag = 0;
    *odd_fills = 0;
    for (int i = 0; i < SOFTMAX_WARPS; ++i) live[i] = -1;   // no key tile's tag
    fence_mbarrier_init();
  }
  if (warp == MMA_WARP) {
    if constexpr (PAIR) {   // one warp in each CTA: the same columns in both
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();   // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint32_t prod_fills = 0;   // ring fills this CTA's producer issued (pair form, producer thread)
  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const CUtensorMap* tm_k = PAIR ? &args.tm_k64 : &args.tm_k;   // a pair CTA loads 64 keys per tile
      tma_prefetch_desc(&args.tm_q);
      tma_prefetch_desc(tm_k);
      tma_prefetch_desc(&args.tm_v);
      // copies into this CTA's shared memory complete on the even CTA's barriers, which
      // count both CTAs' bytes
      const bool arms = rank == 0;
      auto load = [&](uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
        if constexpr (PAIR) tma_load_3d_pair(dst, map, mapa_shared(smem_u32(bar), 0), c0, c1, bh);
        else tma_load_3d(dst, map, bar, c0, c1, bh);
      };
      if (arms) mbar_arrive_expect_tx(q_full, NCTA * NGROUP * C::TILE_BYTES);
      for (int g = 0; g < NGROUP; ++g)
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          load(sQ + g * C::TILE_BYTES + c * BOX_BYTES, &args.tm_q, q_full, c * 64, tile_row0(g, rank));
      uint32_t it = 0;
      uint32_t last_par[NST];
      bool issued[NST];
#pragma unroll
      for (int i = 0; i < NST; ++i) {
        issued[i] = false;
        last_par[i] = 0;
      }
      auto issue = [&](bool is_v, int j) -> bool {
        const int st = it % NST;
        const uint32_t par = (it / NST) & 1u;
        if (!wait_bar(&ring_empty[st], par ^ 1u)) return false;
        if (arms) mbar_arrive_expect_tx(&ring_full[st], NCTA * C::STAGE_BYTES);
        uint8_t* dst = sRing + st * C::STAGE_BYTES;
        if (PAIR && is_v) {
          load(dst, &args.tm_v, &ring_full[st], static_cast<int>(rank) * 64, j * BN);   // 64 columns, 128 keys
        } else {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            load(dst + c * (PAIR ? HALF_BOX_BYTES : BOX_BYTES), is_v ? &args.tm_v : tm_k, &ring_full[st], c * 64,
                 j * BN + static_cast<int>(rank) * (BN / NCTA));
        }
        issued[st] = true;
        last_par[st] = par;
        ++it;
        return true;
      };
      bool ok = true;
      // pass 1: K of every tile either product takes; pass 2 over those tiles t0 < t1 < ...:
      // K_t0, then K_ti and V_t(i-1) interleaved, then the last V
      uint32_t uw = ~0u;   // tiles either product takes (unmasked: all nkt)
      for (int j = 0; j < nkt && ok; ++j) {
        if constexpr (MASK) {
          if ((j & 31) == 0) uw = union_word(j >> 5);
          if (!bit(uw, j)) continue;
        }
        ok = issue(false, j);
      }
      int prev = -1;
      for (int j = 0; j < nkt && ok; ++j) {
        if constexpr (MASK) {
          if ((j & 31) == 0) uw = union_word(j >> 5);
          if (!bit(uw, j)) continue;
        }
        ok = issue(false, j);
        if (ok && prev >= 0) ok = issue(true, prev);
        prev = j;
      }
      if (ok && prev >= 0) ok = issue(true, prev);
      if constexpr (PAIR) {
        // Both CTAs' copies complete on the even CTA's barriers, so the even producer drains
        // them for both, after the first closing cluster barrier.  The two producers may have
        // stopped after different numbers of fills (each gives up on its own CTA's abort flag
        // or wait limit), so the odd one publishes its count for the even one to settle.
        prod_fills = it;
        if (rank != 0) st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(odd_fills)), 0), it);
      } else {
        drain_wait(q_full, 0, ctx);
        for (int i = 0; i < NST; ++i)
          if (issued[i]) drain_wait(&ring_full[i], last_par[i], ctx);
      }
    }
  } else if (warp >= MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuers
    // One thread per query tile g issues S_g and O_g products and does its own waits:
    // a wait costs the issuing thread a few hundred cycles, and with two issuers the
    // tensor core runs the other tile's queued products meanwhile.  In a pair only the
    // even CTA issues; the odd CTA's issuer warps only hold its tensor memory.
    const int g = warp - MMA_WARP;
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(NCTA * BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_fp16_f32(NCTA * BM, D, 0, 1);   // P and V in fp16
      // bytes per 64-column atom of this CTA's K rows (128 keys, or 64 in a pair)
      constexpr int KATOM = PAIR ? HALF_BOX_BYTES : BOX_BYTES;
      auto mma = [&](uint32_t d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
        if constexpr (PAIR) tc_mma_f16_pair(d, a_desc, b_desc, idesc, acc);
        else tc_mma_f16(d, a_desc, b_desc, idesc, acc);
      };
      const uint32_t sRa = smem_u32(sRing);
      // descriptors as (low word + offset / 16, constant high word): one add per operand
      constexpr uint32_t HI = sdesc_hi_sw128(1024);
      const uint32_t qlo = sdesc_lo(smem_u32(sQ) + g * C::TILE_BYTES, 16);
      const uint32_t plo = sdesc_lo(smem_u32(sP) + g * C::P_BYTES, 16);
      const uint32_t scol = tmem + TMEM_S + g * 128;
      const uint32_t ocol = tmem + TMEM_O + g * 128;
      // key tiles each query tile of product g can see (0 for a tile wholly past N_Q):
      // only those count as visited (query tile, key tile) pairs
      auto tile_keys = [&](int r, int n) {
        const int r0 = tile_row0(g, r);
        return r0 < s.NQ ? (s.causal ? min(n - 1, min(s.NQ - 1, r0 + BM - 1)) : n - 1) / BN + 1 : 0;
      };
      const int nkt_a = tile_keys(0, nk);
      const int nkt_b = PAIR ? tile_keys(1, nk) : 0;
      uint32_t pos = 0;   // ring position (K and V tiles in producer order)
      uint32_t uc0 = 0, uc1 = 0;   // S products issued into score buffer 0 and 1
      // pairs in the product's range (its query tiles' key ranges over all N_K keys: those
      // past nk, of an item run over fewer keys, count as skipped), and those whose P V
      // product ran
      const unsigned long long visited =
          static_cast<unsigned long long>(tile_keys(0, s.NK) + (PAIR ? tile_keys(1, s.NK) : 0));
      unsigned long long ran = 0;
      bool o_started = false;
      auto ring_wait = [&](uint32_t p, uint32_t& addr) -> bool {
        const int st = p % NST;
        if (!wait_bar(&ring_full[st], (p / NST) & 1u)) return false;
        tc_fence_after();
        addr = sRa + st * C::STAGE_BYTES;
        return true;
      };
      // S_g = Q_g K^T into score buffer b (buffer 1 exists in pass 1 only: it is the O_g
      // region, free until the first O_g product of pass 2)
      auto mma_s = [&](uint32_t kaddr, int b) -> bool {
        const uint32_t use = b ? uc1 : uc0;
        if (!wait_bar(&s_empty[2 * g + b], (use & 1u) ^ 1u)) return false;
        tc_fence_after();
        const uint32_t klo = sdesc_lo(kaddr, 16);
        const uint32_t dcol = scol + 256u * b;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qoff = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;
          const uint32_t koff = ((kk >> 2) * KATOM + (kk & 3) * 32) >> 4;
          mma(dcol, sdesc(qlo + qoff, HI), sdesc(klo + koff, HI), idesc_qk, kk > 0 ? 1u : 0u);
        }
        commit(&s_full[2 * g + b]);
        if (b) ++uc1; else ++uc0;
        return true;
      };
      // O_g += P_g V_j, the product's c-th P tile (p_full's phase c)
      auto mma_pv = [&](int j, uint32_t c, uint32_t vaddr) -> bool {
        if (!wait_bar(&p_full[g], c & 1u)) return false;   // P tiles and votes of both CTAs
        tc_fence_after();
        // votes of the warps of product g (the odd CTA's read from its shared memory), each
        // tagged with its key tile: a vote that is not this tile's counts as live, so the
        // product is skipped only when every vote is current and dead
        int v[NCTA * GROUP_WARPS];
#pragma unroll
        for (int w = 0; w < GROUP_WARPS; ++w) v[w] = live[g * GROUP_WARPS + w];
        if constexpr (PAIR) {
          const uint4 o = ld_shared_cluster_v4(mapa_shared(smem_u32(const_cast<int*>(&live[g * GROUP_WARPS])), 1));
          v[4] = static_cast<int>(o.x);
          v[5] = static_cast<int>(o.y);
          v[6] = static_cast<int>(o.z);
          v[7] = static_cast<int>(o.w);
        }
        int any = 0;
#pragma unroll
        for (int w = 0; w < NCTA * GROUP_WARPS; ++w) any |= (v[w] >> 1) != j || (v[w] & 1);
        if (any != 0) {
          ran += (j < nkt_a ? 1 : 0) + (j < nkt_b ? 1 : 0);   // (query tile, key tile) pairs of the product
          const uint32_t vlo = sdesc_lo(vaddr, BOX_BYTES);
          const uint32_t acc0 = o_started ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t aoff = ((kk >> 2) * BOX_BYTES + (kk & 3) * 32) >> 4;   // P: K-major, 16 keys = 32 B
            const uint32_t boff = (kk * 16 * 128) >> 4;                            // V: MN-major, 16 key rows
            mma(ocol, sdesc(plo + aoff, HI), sdesc(vlo + boff, HI), idesc_pv, kk > 0 ? 1u : acc0);
          }
          o_started = true;
        }
        commit(&p_empty[g]);
        return true;
      };
      bool ok = wait_bar(q_full, 0);
      // test knob: nothing is committed to `drain` yet, so this wait can only time out
      if (ok && ctx.force_timeout) ok = wait_bar(&drain[g], 0);
      uint32_t ka = 0, va = 0;
      // pass 1: S_g(j) for every key tile the product takes, into score buffer c & 1 for its
      // c-th; a ring stage is free once both issuers commit.  Tiles only the other product
      // takes are waited for and released: waiting for the fill keeps this issuer from
      // releasing a stage's next use before the other issuer has read it.
      const int nkt_g = group_keys(g);
      uint32_t uw = ~0u, ow = ~0u;   // tiles either product takes, and this one
      auto refresh = [&](int j) {
        if ((j & 31) == 0) {
          uw = 0;
#pragma unroll
          for (int h = 0; h < NGROUP; ++h) {
            const uint32_t t = take_word(h, j >> 5);
            uw |= t;
            if (h == g) ow = t;
          }
        }
      };
      uint32_t c = 0;
      for (int j = 0; j < nkt && ok; ++j) {
        if constexpr (MASK) {
          refresh(j);
          if (!bit(uw, j)) continue;
        }
        const bool mine = MASK ? bit(ow, j) : j < nkt_g;
        ok = ring_wait(pos, ka);
        if (ok && mine) ok = mma_s(ka, static_cast<int>(c++ & 1u));
        if (ok) commit(&ring_empty[pos % NST]);
        ++pos;
      }
      // pass 2 over the same tiles t0 < t1 < ...: S_g(t0); then per ti, i >= 1: S_g(ti),
      // O_g(t(i-1)); then O_g of the last.  Every S product into buffer 0; the c-th O product
      // after the c-th P tile
      c = 0;
      int prev = -1;
      bool prev_mine = false;
      for (int j = 0; j < nkt && ok; ++j) {
        if constexpr (MASK) {
          refresh(j);
          if (!bit(uw, j)) continue;
        }
        const bool mine = MASK ? bit(ow, j) : j < nkt_g;
        const uint32_t kpos = pos++;
        ok = ring_wait(kpos, ka);
        if (ok && mine) ok = mma_s(ka, 0);
        if (ok) commit(&ring_empty[kpos % NST]);
        if (ok && prev >= 0) {
          const uint32_t vpos = pos++;
          ok = ring_wait(vpos, va);
          if (ok && prev_mine) ok = mma_pv(prev, c++, va);
          if (ok) commit(&ring_empty[vpos % NST]);
        }
        prev = j;
        prev_mine = mine;
      }
      if (ok && prev >= 0) {
        const uint32_t vpos = pos++;
        ok = ring_wait(vpos, va);
        if (ok && prev_mine) ok = mma_pv(prev, c++, va);
        if (ok) commit(&ring_empty[vpos % NST]);
      }
      if (ok) commit(&o_full[g]);
      commit(&drain[g]);
      drain_wait(&drain[g], 0, ctx);
      if (ok && args.tile_counts) {
        atomicAdd(&args.tile_counts[0], visited);
        atomicAdd(&args.tile_counts[1], visited - ran);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    // Warp w serves query tile g = w / 4 and TMEM lanes 32 (w % 4) .. + 31 (its rows).
    const int g = warp / GROUP_WARPS;
    const int quarter = warp % GROUP_WARPS;
    const int row_local = quarter * 32 + lane;   // TMEM lane
    const int row = tile_row0(g, static_cast<int>(rank)) + row_local;
    const int lim = s.causal ? min(row, nk - 1) : nk - 1;   // last key this row may see
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t scol = lane_addr + TMEM_S + g * 128;
    auto warp_wait = [&](uint64_t* bar, uint32_t par) -> bool {
      int r = 1;
      if (lane == 0) r = wait_bar(bar, par) ? 1 : 0;
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    // this row's attention-mask words: four per key tile (rows past N_Q read the last row)
    const uint32_t* mrow = nullptr;
    if (MASK) {
      const int gm = (args.mask.mb > 1 ? bh / s.H : 0) * args.mask.mh + (args.mask.mh > 1 ? bh % s.H : 0);
      mrow = args.mask.bits + (static_cast<size_t>(gm) * s.NQ + min(row, s.NQ - 1)) * args.mask.words;
    }
    auto mask_words = [&](int j, uint32_t (&mw)[4]) {
      if (MASK) {
        const uint4 u = *reinterpret_cast<const uint4*>(mrow + 4 * j);
        mw[0] = u.x;
        mw[1] = u.y;
        mw[2] = u.z;
        mw[3] = u.w;
      } else {
        mw[0] = mw[1] = mw[2] = mw[3] = ~0u;
      }
    };
    uint32_t sv[BN / 32][32];
    // S_g into registers, then hand the buffer back to the MMA thread
    auto take_s = [&](int b, uint32_t use) -> bool {
      if (!warp_wait(&s_full[2 * g + b], use & 1u)) return false;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < BN / 32; ++k) tmem_ld32(scol + 256u * b + 32 * k, sv[k]);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_even(&s_empty[2 * g + b]);
      return true;
    };
#define SV(c) u2f(sv[(c) >> 5][(c) & 31])

    bool ok = true;
    uint32_t sidx = 0;
    float m = -INFINITY;
    int a = -1;
    int jm = 0;   // 32-column chunk (tile * 4 + chunk) holding the first occurrence of the maximum
    // pass 1: running maximum of the raw scores q.k (scale > 0 keeps the argmax), over the
    // key tiles the product takes; its c-th sits in score buffer c & 1, as that buffer's use c >> 1
    uint32_t c = 0;
    const int nkt_g = group_keys(g);
    uint32_t tw = 0;   // tiles this product takes (masked instances), refreshed every 32
    for (int j = 0; j < nkt_g && ok; ++j) {
      if constexpr (MASK) {
        if ((j & 31) == 0) tw = take_word(g, j >> 5);
        if (!bit(tw, j)) continue;
      }
      uint32_t mw[4];
      mask_words(j, mw);   // issued before the wait below: its latency hides behind it
      ok = take_s(static_cast<int>(c & 1u), c >> 1);
      ++c;
      if (!ok) break;
      const int col0 = j * BN;   // key index of column 0
      // maximum of each 32-column chunk; the first chunk (in key order) that raises the
      // running maximum strictly is remembered, so ties keep the lowest index
      float cm[BN / 32];
      if (!MASK && col0 + BN - 1 <= lim) {
#pragma unroll
        for (int k = 0; k < BN / 32; ++k) {
          float u0 = -INFINITY, u1 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            u0 = max3f(u0, u2f(sv[k][c]), u2f(sv[k][c + 1]));
            u1 = max3f(u1, u2f(sv[k][c + 2]), u2f(sv[k][c + 3]));
          }
          cm[k] = fmaxf(u0, u1);
        }
      } else {
#pragma unroll
        for (int k = 0; k < BN / 32; ++k) {
          float u0 = -INFINITY, u1 = -INFINITY;
          // With an attention mask this branch is taken by the whole warp (the condition above
          // is false for every lane), so the chunk vote is safe: a chunk every row of the warp
          // may see whole takes the plain max, a chunk none of them may see is skipped (key
          // padding and block masks are uniform per chunk).  Without one, the branch is taken
          // per lane on causal diagonal tiles and must hold no warp vote: every chunk is mixed.
          int kind = kChunkMixed;
          if constexpr (MASK) kind = chunk_kind(mw[k], col0 + 32 * k, lim);
          if (kind == kChunkAll) {
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              u0 = max3f(u0, u2f(sv[k][c]), u2f(sv[k][c + 1]));
              u1 = max3f(u1, u2f(sv[k][c + 2]), u2f(sv[k][c + 3]));
            }
          } else if (kind == kChunkMixed) {
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              u0 = fmaxf(u0, (col0 + 32 * k + c <= lim && ((mw[k] >> c) & 1u)) ? u2f(sv[k][c]) : -INFINITY);
              u1 = fmaxf(u1, (col0 + 32 * k + c + 1 <= lim && ((mw[k] >> (c + 1)) & 1u)) ? u2f(sv[k][c + 1])
                                                                                         : -INFINITY);
            }
          }
          cm[k] = fmaxf(u0, u1);
        }
      }
#pragma unroll
      for (int k = 0; k < BN / 32; ++k) {
        jm = (cm[k] > m) ? (j * (BN / 32) + k) : jm;
        m = fmaxf(m, cm[k]);
      }
    }

    // pass 2: phi, sum(phi), P tiles.  Per tile: the first 64 columns are loaded and their
    // phi formed in registers; the second 64 columns are loaded and the score buffer handed
    // back; then, once the previous product has released the P tile, both halves are stored.
    const float m_sc = m * s.scale;
    const float c2 = s.scale * (1.0f / 32.0f);
    // a row with no visible key (possible under an attention mask) keeps m = -inf: base 2
    // then saturates every w to 1 (phi = 0), and the row's output is 0
    const float base = (m > -INFINITY) ? fmaf(m_sc, 1.0f / 32.0f, 0.5f) : 2.0f;
    uint8_t* prow = sP + g * C::P_BYTES + row_local * 128;
    float rowsum = 0.0f;
    sidx = (c + 1) >> 1;   // pass 1 used buffer 0 for its tiles 0, 2, 4, ...
    c = 0;                 // P tiles written
    for (int j = 0; j < nkt_g && ok; ++j) {
      if constexpr (MASK) {
        if ((j & 31) == 0) tw = take_word(g, j >> 5);
        if (!bit(tw, j)) continue;
      }
      uint32_t mw[4];
      mask_words(j, mw);   // in flight during the wait
      ok = warp_wait(&s_full[2 * g], sidx & 1u);   // buffer 0
      if (!ok) break;
      ++sidx;
      tc_fence_after();
      const int col0 = j * BN;
      const bool masked = MASK || col0 + BN - 1 > lim;
      const bool arg_tile = j == (jm >> 2) && m > -INFINITY;
      uint32_t h[2][32];
      tmem_ld32(scol, h[0]);
      tmem_ld32(scol + 32, h[1]);
      tc_wait_ld();
      if (arg_tile && (jm & 3) < 2)   // lowest visible column holding the maximum
        a = col0 + ((jm & 1) ? 32 + find_in_chunk(h[1], m, col0 + 32, lim, mw[1])
                             : find_in_chunk(h[0], m, col0, lim, mw[0]));
      uint32_t pk[32];
      float2 tsum2 = phi_half_any<MASK>(masked, h, pk, col0, lim, c2, base, mw[0], mw[1]);
      tmem_ld32(scol + 64, h[0]);
      tmem_ld32(scol + 96, h[1]);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_even(&s_empty[2 * g]);
      if (arg_tile && (jm & 3) >= 2)
        a = col0 + 64 +
            ((jm & 1) ? 32 + find_in_chunk(h[1], m, col0 + 96, lim, mw[3])
                      : find_in_chunk(h[0], m, col0 + 64, lim, mw[2]));
      // the P tile is free once the previous O_g += P_g V product has completed
      ok = warp_wait(&p_empty[g], (c & 1u) ^ 1u);
      if (!ok) break;
      store_p_half(pk, prow, row_local);
      float2 t2;
      {
        uint32_t pk2[32];
        t2 = phi_half_any<MASK>(masked, h, pk2, col0 + 64, lim, c2, base, mw[2], mw[3]);
        store_p_half(pk2, prow + BOX_BYTES, row_local);
      }
      tsum2 = __fadd2_rn(tsum2, t2);
      fence_proxy_async_smem();
      const float tsum = tsum2.x + tsum2.y;
      const unsigned any_live = __any_sync(0xffffffffu, tsum > 0.0f);
      if (lane == 0) {
        live[g * GROUP_WARPS + quarter] = 2 * j + (any_live ? 1 : 0);
      }
      __syncwarp();
      if (lane == 0) arrive_even(&p_full[g]);
      ++c;
      rowsum += tsum;
    }
#undef SV
    if (ok) ok = warp_wait(&o_full[g], 0);
    if (ok) {
      tc_fence_after();
      const bool row_ok = row < s.NQ;
      const float inv = rowsum > 0.0f ? 1.0f / rowsum : 0.0f;   // 0: a row with no visible key
      const size_t ro = static_cast<size_t>(bh) * s.NQ + (row_ok ? row : 0);
      // O rows leave through this query tile's P tile (free: o_full means the last P V
      // product has read it), 4 KB per warp, in whole row segments
      uint8_t* stage = sP + g * C::P_BYTES + quarter * 4096;
      const int wrow0 = tile_row0(g, static_cast<int>(rank)) + quarter * 32;   // first row of this warp
      const size_t row0 = static_cast<size_t>(bh) * s.NQ + wrow0;
      const int n_ok = max(0, min(32, s.NQ - wrow0));
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        tmem_ld32(lane_addr + TMEM_O + g * 128 + c0, ov);
        tc_wait_ld();
        float o[32];
#pragma unroll
        // a row with no visible key writes exact zeros: when every P V product of the query
        // tile was skipped, the accumulator was never written and holds stale bits
        for (int e = 0; e < 32; ++e) o[e] = rowsum > 0.0f ? u2f(ov[e]) * inv : 0.0f;
        if (args.out_bf16)
          warp_store_block32<true>(stage, o, args.o, row0, D, c0, n_ok, lane);
        else
          warp_store_block32<false>(stage, o, args.o, row0, D, c0, n_ok, lane);
      }
      if (row_ok) {
        if (args.row_m) args.row_m[ro] = m_sc;
        if (args.row_s) args.row_s[ro] = rowsum;
        if (args.row_arg) args.row_arg[ro] = a;
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if constexpr (PAIR) {
    // Every role of both CTAs has stopped issuing, and the odd producer's fill count is
    // visible.  The even producer settles the fills only one CTA issued -- it arms those only
    // the odd CTA issued for the odd CTA's bytes alone, and counts the bytes of the odd CTA's
    // copies that never came for those only it issued -- then drains every fill, so no copy
    // is still landing in either CTA when the memory is freed.  The second barrier keeps both
    // CTAs (their shared memory, barriers and tensor memory) alive until then: a pair's
    // products read both CTAs' shared memory and write both tensor memories.
    cluster_sync();
    if (warp == PRODUCER_WARP && lane == 0 && rank == 0) {
      const uint32_t it_e = prod_fills, it_o = *odd_fills;
      const uint32_t lo = min(it_e, it_o), hi = max(it_e, it_o);
      for (uint32_t f = lo; f < hi; ++f) {
        if (f >= it_e) mbar_arrive_expect_tx(&ring_full[f % NST], C::STAGE_BYTES);
        else mbar_complete_tx(&ring_full[f % NST], C::STAGE_BYTES);
      }
      drain_wait(q_full, 0, ctx);
      for (uint32_t st = 0; st < static_cast<uint32_t>(NST) && st < hi; ++st)
        drain_wait(&ring_full[st], ((hi - 1 - st) / NST) & 1u, ctx);
    }
    cluster_sync();
  }
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, TMEM_COLS);
    else tmem_dealloc(tmem, TMEM_COLS);
  }
}

// The masked instances run an item whose mask is a plain key range (fwd_plain_keys) as an
// unmasked one: same protocol, none of the mask's per-tile work.
template <int D, bool MASK, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_tc_kernel(const AttnShape s, const __grid_constant__ FwdTcArgs args, const LaunchCtx ctx) {
  if constexpr (MASK) {
    int bh, q0;
    fwd_item<PAIR>(s, bh, q0);
    const int nk = fwd_plain_keys<PAIR>(s, args, bh, q0);
    if (nk > 0) {
      fwd_body<D, false, PAIR>(s, args, ctx, nk);
      return;
    }
  }
  fwd_body<D, MASK, PAIR>(s, args, ctx, s.NK);
}

template <int D, bool MASK, bool PAIR>
cudaError_t launch_fwd_d(const AttnShape& s, const FwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st) {
  using C = FwdCfg<D, PAIR>;
  auto kernel = attn_fwd_tc_kernel<D, MASK, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int nqt = (s.NQ + BM - 1) / BM;
  const int nct = (nqt + C::NCTA * NGROUP - 1) / (C::NCTA * NGROUP);
  const unsigned grid = static_cast<unsigned>(nct) * static_cast<unsigned>(s.B * s.H) * C::NCTA;
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, s, a, ctx);
  } else {
    kernel<<<grid, THREADS, C::SMEM_BYTES, st>>>(s, a, ctx);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_attn_fwd_tc(const AttnShape& s, const FwdTcArgs& a, const LaunchCtx& ctx, cudaStream_t st) {
  const bool mask = a.mask.bits != nullptr;
  if (s.D == 128 && a.pair) {
    return mask ? launch_fwd_d<128, true, true>(s, a, ctx, st) : launch_fwd_d<128, false, true>(s, a, ctx, st);
  }
  if (s.D == 128) {
    return mask ? launch_fwd_d<128, true, false>(s, a, ctx, st) : launch_fwd_d<128, false, false>(s, a, ctx, st);
  }
  if (s.D == 64) {
    return mask ? launch_fwd_d<64, true, false>(s, a, ctx, st) : launch_fwd_d<64, false, false>(s, a, ctx, st);
  }
  return cudaErrorInvalidValue;
}


}  // namespace raattn
