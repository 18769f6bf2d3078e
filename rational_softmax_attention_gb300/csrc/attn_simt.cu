// fp32 ra_attention on the CUDA cores (FFMA only, never TF32), forward and backward.
//
// Page "Ra-Family: Rational Neural Architecture", section 3, ra_attention
// (two passes per query tile: row maximum, then phi, sum(phi) and phi V) and
// ra_softmax "Closed-Form Backward Pass".  This path serves fp32 inputs, where
// the required accuracy (2e-5 absolute) rules out reduced-precision tensor cores.
//
// Layout of the work: a group of G = D/32 threads owns one query row (forward,
// dQ) or one key row (dK/dV); thread `part` of a group holds the 4-dimension
// chunks part, part + G, part + 2G, ... (read from shared memory as 16-byte
// loads), so the G partial dot products are summed with G-1 xor shuffles.
// The other operand is staged in shared memory 32 rows at a time.  Scores are
// recomputed with exactly the same operation order in every kernel (the
// register-blocked forward for D = 64 and 128 included), so the argmax entry has
// Delta = 0 exactly in the second pass and in the backward.
#include "kernels.cuh"

namespace raattn {

namespace {

template <int D>
struct SimtGeom {
  static constexpr int G = (D >= 32) ? D / 32 : 1;   // threads per row
  static constexpr int DPT = D / G;                  // dimensions per thread
  static constexpr int THREADS = 128;
  static constexpr int ROWS = THREADS / G;           // rows per CTA
  static constexpr int KT = 32;                      // rows of the other operand per stage
};

// Dimension of local index dl (0 .. DPT-1) of thread `part`: chunk part + G (dl / 4), element dl % 4.
template <int G>
__device__ __forceinline__ int dim_of(int dl, int part) {
  return 4 * (part + G * (dl >> 2)) + (dl & 3);
}

// The DPT values thread `part` holds of a shared-memory row (16-byte aligned), in local order.
template <int D>
__device__ __forceinline__ void load_part(const float* row, int part, float (&out)[SimtGeom<D>::DPT]) {
  constexpr int G = SimtGeom<D>::G;
#pragma unroll
  for (int c = 0; c < SimtGeom<D>::DPT / 4; ++c) {
    const float4 w = *reinterpret_cast<const float4*>(row + 4 * (part + G * c));
    out[4 * c] = w.x;
    out[4 * c + 1] = w.y;
    out[4 * c + 2] = w.z;
    out[4 * c + 3] = w.w;
  }
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = 1; o < G; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float load_val(const void* p, size_t idx, int bf16) {
  return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx])
              : reinterpret_cast<const float*>(p)[idx];
}

__device__ __forceinline__ void store_val(void* p, size_t idx, float val, int bf16) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16*>(p)[idx] = __float2bfloat16_rn(val);
  else
    reinterpret_cast<float*>(p)[idx] = val;
}

// phi(Delta) in IEEE fp32 for Delta < 16: ((1-u)/(1+u))^8 with u = Delta/16.
__device__ __forceinline__ float phi_exact(float delta) {
  const float u = delta * (1.0f / 16.0f);
  const float qq = (1.0f - u) / (1.0f + u);
  const float q2 = qq * qq;
  const float q4 = q2 * q2;
  return q4 * q4;
}

// 1/(1-u^2) with u = Delta/16, as 256 / ((16 - Delta)(16 + Delta)).
__device__ __forceinline__ float inv_one_minus_u2(float delta) {
  return 256.0f / ((16.0f - delta) * (16.0f + delta));
}

template <int D>
__device__ __forceinline__ void stage_rows(float (*dst)[D], const float* src, int row0, int nrows) {
  constexpr int KT = SimtGeom<D>::KT;
  for (int e = threadIdx.x; e < KT * D; e += SimtGeom<D>::THREADS) {
    const int rr = e / D, d = e % D;
    const int row = row0 + rr;
    dst[rr][d] = (row < nrows) ? src[static_cast<size_t>(row) * D + d] : 0.0f;
  }
}

template <int D>
__global__ void __launch_bounds__(128) attn_fwd_simt_kernel(AttnShape s, const float* __restrict__ q,
                                                            const float* __restrict__ k,
                                                            const float* __restrict__ v, void* o, int out_bf16,
                                                            float* row_m, float* row_s, int32_t* row_arg) {
  using Gm = SimtGeom<D>;
  constexpr int G = Gm::G, DPT = Gm::DPT, ROWS = Gm::ROWS, KT = Gm::KT;
  __shared__ __align__(16) float ks[KT][D];
  __shared__ __align__(16) float vs[KT][D];
  const int bh = blockIdx.y;
  const int r = threadIdx.x / G, part = threadIdx.x % G;
  const int i = blockIdx.x * ROWS + r;
  const bool row_ok = i < s.NQ;
  const float* qh = q + static_cast<size_t>(bh) * s.NQ * D;
  const float* kh = k + static_cast<size_t>(bh) * s.NK * D;
  const float* vh = v + static_cast<size_t>(bh) * s.NK * D;

  float qr[DPT];
#pragma unroll
  for (int d = 0; d < DPT; ++d) qr[d] = row_ok ? qh[static_cast<size_t>(i) * D + dim_of<G>(d, part)] : 0.0f;
  const int last_row = min(s.NQ - 1, static_cast<int>(blockIdx.x) * ROWS + ROWS - 1);
  const int kend = s.causal ? min(s.NK, last_row + 1) : s.NK;
  const int lim = s.causal ? min(i, s.NK - 1) : s.NK - 1;   // last key this row may see

  // pass 1: row maximum of the scaled scores, lowest index on ties
  float m = -INFINITY;
  int a = -1;
  for (int j0 = 0; j0 < kend; j0 += KT) {
    __syncthreads();
    stage_rows<D>(ks, kh, j0, s.NK);
    __syncthreads();
    const int jn = min(KT, kend - j0);
    for (int jj = 0; jj < jn; ++jj) {
      float kv[DPT];
      load_part<D>(ks[jj], part, kv);
      float dot = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) dot = fmaf(qr[d], kv[d], dot);
      dot = group_sum<G>(dot);
      const float sc = dot * s.scale;
      const int j = j0 + jj;
      if (j <= lim && sc > m) {
        m = sc;
        a = j;
      }
    }
  }

  // pass 2: phi, sum(phi), phi V
  float acc[DPT];
#pragma unroll
  for (int d = 0; d < DPT; ++d) acc[d] = 0.0f;
  float sum = 0.0f;
  for (int j0 = 0; j0 < kend; j0 += KT) {
    __syncthreads();
    stage_rows<D>(ks, kh, j0, s.NK);
    stage_rows<D>(vs, vh, j0, s.NK);
    __syncthreads();
    const int jn = min(KT, kend - j0);
    for (int jj = 0; jj < jn; ++jj) {
      float kv[DPT];
      load_part<D>(ks[jj], part, kv);
      float dot = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) dot = fmaf(qr[d], kv[d], dot);
      dot = group_sum<G>(dot);
      const float sc = dot * s.scale;
      const int j = j0 + jj;
      const float delta = m - sc;
      if (j <= lim && delta < 16.0f) {
        const float phi = phi_exact(delta);
        sum += phi;
        float vv[DPT];
        load_part<D>(vs[jj], part, vv);
#pragma unroll
        for (int d = 0; d < DPT; ++d) acc[d] = fmaf(phi, vv[d], acc[d]);
      }
    }
  }
  if (row_ok) {
    const size_t ro = static_cast<size_t>(bh) * s.NQ + i;
#pragma unroll
    for (int d = 0; d < DPT; ++d) store_val(o, ro * D + dim_of<G>(d, part), acc[d] / sum, out_bf16);
    if (part == 0) {
      if (row_m) row_m[ro] = m;
      if (row_s) row_s[ro] = sum;
      if (row_arg) row_arg[ro] = a;
    }
  }
}

// Register-blocked forward for D = 64 and 128: a CTA of 256 threads owns 64 query rows and
// streams the keys in tiles of 32.  Thread (ty, tx) holds the scores of rows 4 ty .. 4 ty + 3
// against keys tx and tx + 16 of the tile, and the output block of the same rows and
// dimensions D/16 tx .. + D/16 - 1; operands come from padded shared-memory rows as 16-byte
// loads, several FMAs per load.  Every score keeps the operation order of the group kernels
// (G = D/32 partial sums, partial g over the 4-dimension chunks g, g + G, ... in increasing
// order, combined as a pairwise tree), so the backward's recomputed scores, the row maximum
// and the argmax are bitwise the ones of the group-per-row kernels.
// Rows row0 .. row0 + rows - 1 of a [nrows, D] fp32 matrix into a shared tile with row pitch
// `pitch` floats (16-byte aligned), zeros past nrows; all threads of the block take part.
template <int D>
__device__ __forceinline__ void stage_tile(float* dst, int pitch, const float* src, int row0, int rows, int nrows) {
  for (int e = threadIdx.x; e < rows * (D / 4); e += blockDim.x) {
    const int r = e / (D / 4), c4 = e % (D / 4);
    const int row = row0 + r;
    *reinterpret_cast<float4*>(dst + r * pitch + 4 * c4) =
        row < nrows ? reinterpret_cast<const float4*>(src + static_cast<size_t>(row) * D)[c4]
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
}

// out[r][c] = dot(A row r, B row 16 c) for r < 4, c < 2 (A, B shared tiles with pitches lda,
// ldb), in the group kernels' operation order: partial g over the 4-dimension chunks g,
// g + G, ... in increasing order, the G partials summed as a pairwise tree.
template <int D>
__device__ __forceinline__ void block_dot(const float* A, int lda, const float* B, int ldb, float (&out)[4][2]) {
  constexpr int G = D / 32;
  float p[4][2][G];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int g = 0; g < G; ++g) p[r][c][g] = 0.0f;
#pragma unroll(4 / G)
  for (int d0 = 0; d0 < D / 4; d0 += G) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int d4 = d0 + g;
      float4 a[4], b[2];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4*>(A + r * lda + 4 * d4);
#pragma unroll
      for (int c = 0; c < 2; ++c) b[c] = *reinterpret_cast<const float4*>(B + 16 * c * ldb + 4 * d4);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          p[r][c][g] = fmaf(a[r].x, b[c].x, p[r][c][g]);
          p[r][c][g] = fmaf(a[r].y, b[c].y, p[r][c][g]);
          p[r][c][g] = fmaf(a[r].z, b[c].z, p[r][c][g]);
          p[r][c][g] = fmaf(a[r].w, b[c].w, p[r][c][g]);
        }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 2; ++c)
      out[r][c] = (G == 4) ? (p[r][c][0] + p[r][c][1]) + (p[r][c][2 % G] + p[r][c][3 % G])
                           : p[r][c][0] + p[r][c][1 % G];
}

template <int D>
struct TiledGeom {
  static constexpr int BQ = 64, BK = 32, THREADS = 256;
  static constexpr int DT = D / 16;       // output dimensions per thread
  static constexpr int LDQ = D + 4;       // padded pitch (floats) of the Q and K rows
  static constexpr int LDP = BQ + 4;      // padded pitch of the transposed P tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + BQ * LDQ;
  static constexpr int OFF_V = OFF_K + BK * LDQ;
  static constexpr int OFF_P = OFF_V + BK * D;
  static constexpr int OFF_X = OFF_P + BK * LDP;   // [BQ][16] per-thread partials (max, then sums)
  static constexpr int OFF_XI = OFF_X + BQ * 16;   // [BQ][16] per-thread argmax
  static constexpr int OFF_M = OFF_XI + BQ * 16;   // [BQ] row max, [BQ] row argmax
  static constexpr int FLOATS = OFF_M + 2 * BQ;
  static constexpr int SMEM_BYTES = FLOATS * 4;
  static_assert(D == 64 || D == 128, "tiled CUDA-core forward: D = 64 or 128");
  static_assert(OFF_K % 4 == 0 && OFF_V % 4 == 0 && OFF_P % 4 == 0 && LDQ % 4 == 0 && LDP % 4 == 0, "16-byte rows");
};

template <int D>
__global__ void __launch_bounds__(256, 2) attn_fwd_simt_tiled_kernel(AttnShape s, const float* __restrict__ q,
                                                                  const float* __restrict__ k,
                                                                  const float* __restrict__ v, void* o,
                                                                  int out_bf16, float* row_m, float* row_s,
                                                                  int32_t* row_arg) {
  using T = TiledGeom<D>;
  constexpr int BQ = T::BQ, BK = T::BK, DT = T::DT, LDQ = T::LDQ, LDP = T::LDP;
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* Qs = sm + T::OFF_Q;
  float* Ks = sm + T::OFF_K;
  float* Vs = sm + T::OFF_V;
  float* Ps = sm + T::OFF_P;
  float* Xf = sm + T::OFF_X;
  int* Xi = reinterpret_cast<int*>(sm + T::OFF_XI);
  float* Mrow = sm + T::OFF_M;
  int* Arow = reinterpret_cast<int*>(sm + T::OFF_M + BQ);
  const int bh = blockIdx.y;
  const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
  const int i0 = blockIdx.x * BQ;
  const float* qh = q + static_cast<size_t>(bh) * s.NQ * D;
  const float* kh = k + static_cast<size_t>(bh) * s.NK * D;
  const float* vh = v + static_cast<size_t>(bh) * s.NK * D;

  stage_tile<D>(Qs, LDQ, qh, i0, BQ, s.NQ);
  const int last_row = min(s.NQ - 1, i0 + BQ - 1);
  const int kend = s.causal ? min(s.NK, last_row + 1) : s.NK;
  int lim[4];   // last key each of this thread's rows may see
#pragma unroll
  for (int r = 0; r < 4; ++r) lim[r] = s.causal ? min(i0 + 4 * ty + r, s.NK - 1) : s.NK - 1;

  // scores of rows 4 ty + r against keys tx + 16 c of the staged key tile
  auto scores = [&](float (&sc)[4][2]) {
    block_dot<D>(Qs + 4 * ty * LDQ, LDQ, Ks + tx * LDQ, LDQ, sc);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 2; ++c) sc[r][c] *= s.scale;
  };

  // pass 1: row maximum of the scaled scores, lowest index on ties
  float m[4];
  int a[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = -INFINITY;
    a[r] = -1;
  }
  for (int j0 = 0; j0 < kend; j0 += BK) {
    __syncthreads();
    stage_tile<D>(Ks, LDQ, kh, j0, BK, s.NK);
    __syncthreads();
    float sc[4][2];
    scores(sc);
#pragma unroll
    for (int c = 0; c < 2; ++c) {   // keys tx, then tx + 16: increasing order within the thread
      const int j = j0 + tx + 16 * c;
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (j <= lim[r] && sc[r][c] > m[r]) {
          m[r] = sc[r][c];
          a[r] = j;
        }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    Xf[(4 * ty + r) * 16 + tx] = m[r];
    Xi[(4 * ty + r) * 16 + tx] = a[r];
  }
  __syncthreads();
  if (t < BQ) {   // combine the 16 threads of a row: the maximum, and the lowest index holding it
    float bm = -INFINITY;
    int ba = -1;
    for (int x = 0; x < 16; ++x) {
      const float vm = Xf[t * 16 + x];
      const int va = Xi[t * 16 + x];
      if (vm > bm) {
        bm = vm;
        ba = va;
      } else if (vm == bm && va >= 0 && (ba < 0 || va < ba)) {
        ba = va;
      }
    }
    Mrow[t] = bm;
    Arow[t] = ba;
  }
  __syncthreads();
  float mr[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) mr[r] = Mrow[4 * ty + r];

  // pass 2: phi, sum(phi), phi V (keys in increasing order for every output element)
  float acc[4][DT];
  float psum[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    psum[r] = 0.0f;
#pragma unroll
    for (int d = 0; d < DT; ++d) acc[r][d] = 0.0f;
  }
  for (int j0 = 0; j0 < kend; j0 += BK) {
    __syncthreads();
    stage_tile<D>(Ks, LDQ, kh, j0, BK, s.NK);
    stage_tile<D>(Vs, D, vh, j0, BK, s.NK);
    __syncthreads();
    float sc[4][2];
    scores(sc);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = j0 + tx + 16 * c;
      float ph[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float delta = mr[r] - sc[r][c];
        ph[r] = (j <= lim[r] && delta < 16.0f) ? phi_exact(delta) : 0.0f;
        psum[r] += ph[r];
      }
      *reinterpret_cast<float4*>(Ps + (tx + 16 * c) * LDP + 4 * ty) = make_float4(ph[0], ph[1], ph[2], ph[3]);
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BK; ++kk) {
      const float4 pp = *reinterpret_cast<const float4*>(Ps + kk * LDP + 4 * ty);
      float vv[DT];
#pragma unroll
      for (int e = 0; e < DT / 4; ++e) {
        const float4 w4 = *reinterpret_cast<const float4*>(Vs + kk * D + DT * tx + 4 * e);
        vv[4 * e] = w4.x;
        vv[4 * e + 1] = w4.y;
        vv[4 * e + 2] = w4.z;
        vv[4 * e + 3] = w4.w;
      }
      const float pr[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int d = 0; d < DT; ++d) acc[r][d] = fmaf(pr[r], vv[d], acc[r][d]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) Xf[(4 * ty + r) * 16 + tx] = psum[r];
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = i0 + 4 * ty + r;
    float sum = 0.0f;
    for (int x = 0; x < 16; ++x) sum += Xf[(4 * ty + r) * 16 + x];
    if (row >= s.NQ) continue;
    const size_t ro = static_cast<size_t>(bh) * s.NQ + row;
    const float inv = 1.0f / sum;
#pragma unroll
    for (int d = 0; d < DT; ++d) store_val(o, ro * D + DT * tx + d, acc[r][d] * inv, out_bf16);
    if (tx == 0) {
      if (row_m) row_m[ro] = mr[r];
      if (row_s) row_s[ro] = sum;
      if (row_arg) row_arg[ro] = Arow[4 * ty + r];
    }
  }
}

// dQ, with D_i = dO_i . O_i and R_i = sum_{j != a_i} E_ij written to the workspace.
template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dq_simt_kernel(
    AttnShape s, const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const void* o, int o_bf16, const float* __restrict__ dout, const float* __restrict__ row_m,
    const float* __restrict__ row_s, const int32_t* __restrict__ row_arg, void* dq, int grad_bf16,
    float* ws_d, float* ws_r) {
  using Gm = SimtGeom<D>;
  constexpr int G = Gm::G, DPT = Gm::DPT, ROWS = Gm::ROWS, KT = Gm::KT;
  __shared__ __align__(16) float ks[KT][D];
  __shared__ __align__(16) float vs[KT][D];
  const int bh = blockIdx.y;
  const int r = threadIdx.x / G, part = threadIdx.x % G;
  const int i = blockIdx.x * ROWS + r;
  const bool row_ok = i < s.NQ;
  const int ic = row_ok ? i : s.NQ - 1;
  const size_t ro = static_cast<size_t>(bh) * s.NQ + ic;
  const float* kh = k + static_cast<size_t>(bh) * s.NK * D;
  const float* vh = v + static_cast<size_t>(bh) * s.NK * D;

  float qr[DPT], dor[DPT];
  float dpart = 0.0f;
#pragma unroll
  for (int d = 0; d < DPT; ++d) {
    const size_t idx = ro * D + dim_of<G>(d, part);
    qr[d] = q[idx];
    dor[d] = dout[idx];
    dpart = fmaf(dor[d], load_val(o, idx, o_bf16), dpart);
  }
  const float Di = group_sum<G>(dpart);
  const float m = row_m[ro], sum = row_s[ro];
  const int a = row_arg[ro];
  const float inv_sum = 1.0f / sum;
  const int last_row = min(s.NQ - 1, static_cast<int>(blockIdx.x) * ROWS + ROWS - 1);
  const int kend = s.causal ? min(s.NK, last_row + 1) : s.NK;
  const int lim = s.causal ? min(ic, s.NK - 1) : s.NK - 1;

  float acc[DPT];
#pragma unroll
  for (int d = 0; d < DPT; ++d) acc[d] = 0.0f;
  float R = 0.0f;
  for (int j0 = 0; j0 < kend; j0 += KT) {
    __syncthreads();
    stage_rows<D>(ks, kh, j0, s.NK);
    stage_rows<D>(vs, vh, j0, s.NK);
    __syncthreads();
    const int jn = min(KT, kend - j0);
    for (int jj = 0; jj < jn; ++jj) {
      float kv[DPT], vv[DPT];
      load_part<D>(ks[jj], part, kv);
      load_part<D>(vs[jj], part, vv);
      float dot = 0.0f, dp = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) {
        dot = fmaf(qr[d], kv[d], dot);
        dp = fmaf(dor[d], vv[d], dp);
      }
      dot = group_sum<G>(dot);
      dp = group_sum<G>(dp);
      const float sc = dot * s.scale;
      const int j = j0 + jj;
      const float delta = m - sc;
      if (j <= lim && j != a && delta < 16.0f) {
        const float p = phi_exact(delta) * inv_sum;
        const float e = p * (dp - Di) * inv_one_minus_u2(delta);
        R += e;
#pragma unroll
        for (int d = 0; d < DPT; ++d) acc[d] = fmaf(e, kv[d], acc[d]);
      }
    }
  }
  if (row_ok) {
#pragma unroll
    for (int d = 0; d < DPT; ++d) {
      const float ka = kh[static_cast<size_t>(a) * D + dim_of<G>(d, part)];
      store_val(dq, ro * D + dim_of<G>(d, part), s.scale * fmaf(-R, ka, acc[d]), grad_bf16);
    }
    if (part == 0) {
      ws_d[ro] = Di;
      ws_r[ro] = R;
    }
  }
}

// dK and dV, key-major; reads D_i and R_i from the workspace.
template <int D>
__global__ void __launch_bounds__(128) attn_bwd_dkdv_simt_kernel(
    AttnShape s, const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dout, const float* __restrict__ row_m, const float* __restrict__ row_s,
    const int32_t* __restrict__ row_arg, void* dk, void* dv, int grad_bf16, const float* __restrict__ ws_d,
    const float* __restrict__ ws_r) {
  using Gm = SimtGeom<D>;
  constexpr int G = Gm::G, DPT = Gm::DPT, ROWS = Gm::ROWS, KT = Gm::KT;
  __shared__ __align__(16) float qs[KT][D];
  __shared__ __align__(16) float dos[KT][D];
  __shared__ float st_m[KT], st_inv[KT], st_d[KT], st_r[KT];
  __shared__ int st_a[KT];
  const int bh = blockIdx.y;
  const int r = threadIdx.x / G, part = threadIdx.x % G;
  const int j = blockIdx.x * ROWS + r;
  const bool key_ok = j < s.NK;
  const int jc = key_ok ? j : s.NK - 1;
  const size_t ko = static_cast<size_t>(bh) * s.NK + jc;
  const float* qh = q + static_cast<size_t>(bh) * s.NQ * D;
  const float* doh = dout + static_cast<size_t>(bh) * s.NQ * D;
  const size_t so = static_cast<size_t>(bh) * s.NQ;

  float kr[DPT], vr[DPT], adk[DPT], adv[DPT];
#pragma unroll
  for (int d = 0; d < DPT; ++d) {
    kr[d] = k[ko * D + dim_of<G>(d, part)];
    vr[d] = v[ko * D + dim_of<G>(d, part)];
    adk[d] = 0.0f;
    adv[d] = 0.0f;
  }
  const int istart = s.causal ? static_cast<int>(blockIdx.x) * ROWS : 0;   // first query any key here sees
  for (int i0 = istart; i0 < s.NQ; i0 += KT) {
    __syncthreads();
    stage_rows<D>(qs, qh, i0, s.NQ);
    stage_rows<D>(dos, doh, i0, s.NQ);
    if (threadIdx.x < KT) {
      const int ii = i0 + threadIdx.x;
      const bool ok = ii < s.NQ;
      st_m[threadIdx.x] = ok ? row_m[so + ii] : 0.0f;
      st_inv[threadIdx.x] = ok ? 1.0f / row_s[so + ii] : 0.0f;
      st_d[threadIdx.x] = ok ? ws_d[so + ii] : 0.0f;
      st_r[threadIdx.x] = ok ? ws_r[so + ii] : 0.0f;
      st_a[threadIdx.x] = ok ? row_arg[so + ii] : -1;
    }
    __syncthreads();
    const int in = min(KT, s.NQ - i0);
    for (int ii = 0; ii < in; ++ii) {
      float qv[DPT], dov[DPT];
      load_part<D>(qs[ii], part, qv);
      load_part<D>(dos[ii], part, dov);
      float dot = 0.0f, dp = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) {
        dot = fmaf(qv[d], kr[d], dot);
        dp = fmaf(dov[d], vr[d], dp);
      }
      dot = group_sum<G>(dot);
      dp = group_sum<G>(dp);
      const int i = i0 + ii;
      const float sc = dot * s.scale;
      const float delta = st_m[ii] - sc;
      const bool allowed = key_ok && (!s.causal || j <= i);
      if (allowed && delta < 16.0f) {
        const float p = phi_exact(delta) * st_inv[ii];
        const float ds = (j == st_a[ii]) ? -st_r[ii] : p * (dp - st_d[ii]) * inv_one_minus_u2(delta);
#pragma unroll
        for (int d = 0; d < DPT; ++d) {
          adk[d] = fmaf(ds, qv[d], adk[d]);
          adv[d] = fmaf(p, dov[d], adv[d]);
        }
      }
    }
  }
  if (key_ok) {
#pragma unroll
    for (int d = 0; d < DPT; ++d) {
      store_val(dk, ko * D + dim_of<G>(d, part), s.scale * adk[d], grad_bf16);
      store_val(dv, ko * D + dim_of<G>(d, part), adv[d], grad_bf16);
    }
  }
}

// Register-blocked backward for D = 64 and 128, the same blocking as the forward.
//   dQ kernel: 64 query rows per CTA against 32-key tiles; thread (ty, tx) forms the scores
//   and dP of rows 4 ty .. + 3 against keys tx, tx + 16 (block_dot: the forward's scores
//   bitwise), E into a shared tile, then its 4 x D/16 block of dQ += E K; D_i and R_i go to
//   the workspace for the dK/dV kernel.
//   dK/dV kernel: 64 keys per CTA against 32-query tiles; thread (ty, tx) forms S^T and dP^T
//   of keys 4 ty .. + 3 against queries tx, tx + 16, P and dS into shared tiles, then its
//   4 x D/16 blocks of dV += P^T dO and dK += dS^T Q.
// Every output element accumulates over the other operand's rows in increasing order.
template <int D>
struct TiledBwdGeom {
  static constexpr int BR = 64, BT = 32, THREADS = 256, DT = D / 16;
  static constexpr int LDT = D + 4;    // padded pitch of the streamed tiles (read by 16 rows per warp)
  static constexpr int LDE = BR + 4;   // padded pitch of the E / P / dS tiles
  // dQ kernel: Q, dO [BR][D]; K, V [BT][LDT]; E^T [BT][LDE]; R partials [BR][16]; m, 1/s, D_i, a [4][BR]
  static constexpr int DQ_Q = 0, DQ_DO = BR * D, DQ_K = 2 * BR * D, DQ_V = DQ_K + BT * LDT;
  static constexpr int DQ_E = DQ_V + BT * LDT, DQ_X = DQ_E + BT * LDE, DQ_C = DQ_X + BR * 16;
  static constexpr int DQ_BYTES = (DQ_C + 4 * BR) * 4;
  // dK/dV kernel: K, V [BR][D]; Q, dO [BT][LDT]; P, dS [BT][LDE]; m, 1/s, D_i, R_i, a [5][BT]
  static constexpr int KV_K = 0, KV_V = BR * D, KV_Q = 2 * BR * D, KV_DO = KV_Q + BT * LDT;
  static constexpr int KV_P = KV_DO + BT * LDT, KV_S = KV_P + BT * LDE, KV_C = KV_S + BT * LDE;
  static constexpr int KV_BYTES = (KV_C + 5 * BT) * 4;
  static_assert(D == 64 || D == 128, "tiled CUDA-core backward: D = 64 or 128");
  static_assert(DQ_K % 4 == 0 && DQ_V % 4 == 0 && DQ_E % 4 == 0 && KV_Q % 4 == 0 && KV_DO % 4 == 0 &&
                    KV_P % 4 == 0 && KV_S % 4 == 0 && LDT % 4 == 0 && LDE % 4 == 0,
                "16-byte rows");
};

template <int D>
__global__ void __launch_bounds__(256, 2) attn_bwd_dq_simt_tiled_kernel(
    AttnShape s, const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const void* o, int o_bf16, const float* __restrict__ dout, const float* __restrict__ row_m,
    const float* __restrict__ row_s, const int32_t* __restrict__ row_arg, void* dq, int grad_bf16,
    float* ws_d, float* ws_r) {
  using T = TiledBwdGeom<D>;
  constexpr int BR = T::BR, BT = T::BT, DT = T::DT, LDT = T::LDT, LDE = T::LDE;
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* Qs = sm + T::DQ_Q;
  float* Ds = sm + T::DQ_DO;
  float* Ks = sm + T::DQ_K;
  float* Vs = sm + T::DQ_V;
  float* Es = sm + T::DQ_E;
  float* Xf = sm + T::DQ_X;
  float* Cm = sm + T::DQ_C;
  float* Cinv = Cm + BR;
  float* Cd = Cm + 2 * BR;
  int* Ca = reinterpret_cast<int*>(Cm + 3 * BR);
  const int bh = blockIdx.y;
  const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
  const int i0 = blockIdx.x * BR;
  const float* kh = k + static_cast<size_t>(bh) * s.NK * D;
  const float* vh = v + static_cast<size_t>(bh) * s.NK * D;
  stage_tile<D>(Qs, D, q + static_cast<size_t>(bh) * s.NQ * D, i0, BR, s.NQ);
  stage_tile<D>(Ds, D, dout + static_cast<size_t>(bh) * s.NQ * D, i0, BR, s.NQ);
  __syncthreads();
  if (t < BR) {   // per-row constants; D_i = dO_i . O_i
    const int i = i0 + t;
    float m = 0.0f, inv = 0.0f, di = 0.0f;
    int a = -1;
    if (i < s.NQ) {
      const size_t ro = static_cast<size_t>(bh) * s.NQ + i;
      m = row_m[ro];
      inv = 1.0f / row_s[ro];
      a = row_arg[ro];
      for (int d = 0; d < D; ++d) di = fmaf(Ds[t * D + d], load_val(o, ro * D + d, o_bf16), di);
    }
    Cm[t] = m;
    Cinv[t] = inv;
    Cd[t] = di;
    Ca[t] = a;
  }
  __syncthreads();
  float mr[4], invr[4], dr[4];
  int ar[4], lim[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = 4 * ty + r;
    mr[r] = Cm[row];
    invr[r] = Cinv[row];
    dr[r] = Cd[row];
    ar[r] = Ca[row];
    lim[r] = s.causal ? min(i0 + row, s.NK - 1) : s.NK - 1;
  }
  const int last_row = min(s.NQ - 1, i0 + BR - 1);
  const int kend = s.causal ? min(s.NK, last_row + 1) : s.NK;
  float acc[4][DT];
  float rpart[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    rpart[r] = 0.0f;
#pragma unroll
    for (int d = 0; d < DT; ++d) acc[r][d] = 0.0f;
  }
  for (int j0 = 0; j0 < kend; j0 += BT) {
    __syncthreads();
    stage_tile<D>(Ks, LDT, kh, j0, BT, s.NK);
    stage_tile<D>(Vs, LDT, vh, j0, BT, s.NK);
    __syncthreads();
    float sc[4][2], dp[4][2];
    block_dot<D>(Qs + 4 * ty * D, D, Ks + tx * LDT, LDT, sc);
    block_dot<D>(Ds + 4 * ty * D, D, Vs + tx * LDT, LDT, dp);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = j0 + tx + 16 * c;
      float e4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float delta = mr[r] - sc[r][c] * s.scale;
        float e = 0.0f;
        if (j <= lim[r] && j != ar[r] && delta < 16.0f) {
          const float p = phi_exact(delta) * invr[r];
          e = p * (dp[r][c] - dr[r]) * inv_one_minus_u2(delta);
        }
        rpart[r] += e;
        e4[r] = e;
      }
      *reinterpret_cast<float4*>(Es + (tx + 16 * c) * LDE + 4 * ty) = make_float4(e4[0], e4[1], e4[2], e4[3]);
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BT; ++kk) {
      const float4 e4 = *reinterpret_cast<const float4*>(Es + kk * LDE + 4 * ty);
      float kv[DT];
#pragma unroll
      for (int x = 0; x < DT / 4; ++x) {
        const float4 w = *reinterpret_cast<const float4*>(Ks + kk * LDT + DT * tx + 4 * x);
        kv[4 * x] = w.x;
        kv[4 * x + 1] = w.y;
        kv[4 * x + 2] = w.z;
        kv[4 * x + 3] = w.w;
      }
      const float er[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int d = 0; d < DT; ++d) acc[r][d] = fmaf(er[r], kv[d], acc[r][d]);
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) Xf[(4 * ty + r) * 16 + tx] = rpart[r];
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = i0 + 4 * ty + r;
    float R = 0.0f;
    for (int x = 0; x < 16; ++x) R += Xf[(4 * ty + r) * 16 + x];
    if (row >= s.NQ) continue;
    const size_t ro = static_cast<size_t>(bh) * s.NQ + row;
#pragma unroll
    for (int d = 0; d < DT; ++d) {
      const float ka = kh[static_cast<size_t>(ar[r]) * D + DT * tx + d];
      store_val(dq, ro * D + DT * tx + d, s.scale * fmaf(-R, ka, acc[r][d]), grad_bf16);
    }
    if (tx == 0) {
      ws_d[ro] = dr[r];
      ws_r[ro] = R;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256, 1) attn_bwd_dkdv_simt_tiled_kernel(
    AttnShape s, const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dout, const float* __restrict__ row_m, const float* __restrict__ row_s,
    const int32_t* __restrict__ row_arg, void* dk, void* dv, int grad_bf16, const float* __restrict__ ws_d,
    const float* __restrict__ ws_r) {
  using T = TiledBwdGeom<D>;
  constexpr int BR = T::BR, BT = T::BT, DT = T::DT, LDT = T::LDT, LDE = T::LDE;
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* Ks = sm + T::KV_K;
  float* Vs = sm + T::KV_V;
  float* Qt = sm + T::KV_Q;
  float* Dt = sm + T::KV_DO;
  float* Pt = sm + T::KV_P;
  float* St = sm + T::KV_S;
  float* Cm = sm + T::KV_C;
  float* Cinv = Cm + BT;
  float* Cd = Cm + 2 * BT;
  float* Cr = Cm + 3 * BT;
  int* Ca = reinterpret_cast<int*>(Cm + 4 * BT);
  const int bh = blockIdx.y;
  const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
  const int j0 = blockIdx.x * BR;   // first key of the block
  const float* qh = q + static_cast<size_t>(bh) * s.NQ * D;
  const float* doh = dout + static_cast<size_t>(bh) * s.NQ * D;
  const size_t so = static_cast<size_t>(bh) * s.NQ;
  stage_tile<D>(Ks, D, k + static_cast<size_t>(bh) * s.NK * D, j0, BR, s.NK);
  stage_tile<D>(Vs, D, v + static_cast<size_t>(bh) * s.NK * D, j0, BR, s.NK);
  float adk[4][DT], adv[4][DT];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int d = 0; d < DT; ++d) {
      adk[r][d] = 0.0f;
      adv[r][d] = 0.0f;
    }
  const int istart = s.causal ? j0 : 0;   // first query any key of the block sees (j <= i)
  for (int i0 = istart; i0 < s.NQ; i0 += BT) {
    __syncthreads();
    stage_tile<D>(Qt, LDT, qh, i0, BT, s.NQ);
    stage_tile<D>(Dt, LDT, doh, i0, BT, s.NQ);
    if (t < BT) {
      const int ii = i0 + t;
      const bool ok = ii < s.NQ;
      Cm[t] = ok ? row_m[so + ii] : 0.0f;
      Cinv[t] = ok ? 1.0f / row_s[so + ii] : 0.0f;
      Cd[t] = ok ? ws_d[so + ii] : 0.0f;
      Cr[t] = ok ? ws_r[so + ii] : 0.0f;
      Ca[t] = ok ? row_arg[so + ii] : -1;
    }
    __syncthreads();
    float sc[4][2], dp[4][2];
    block_dot<D>(Ks + 4 * ty * D, D, Qt + tx * LDT, LDT, sc);   // S^T: keys x queries
    block_dot<D>(Vs + 4 * ty * D, D, Dt + tx * LDT, LDT, dp);   // dP^T
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int qi = tx + 16 * c;
      const int i = i0 + qi;
      float p4[4], s4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = j0 + 4 * ty + r;
        const float delta = Cm[qi] - sc[r][c] * s.scale;
        const bool allowed = j < s.NK && i < s.NQ && (!s.causal || j <= i);
        float p = 0.0f, ds = 0.0f;
        if (allowed && delta < 16.0f) {
          p = phi_exact(delta) * Cinv[qi];
          ds = (j == Ca[qi]) ? -Cr[qi] : p * (dp[r][c] - Cd[qi]) * inv_one_minus_u2(delta);
        }
        p4[r] = p;
        s4[r] = ds;
      }
      *reinterpret_cast<float4*>(Pt + qi * LDE + 4 * ty) = make_float4(p4[0], p4[1], p4[2], p4[3]);
      *reinterpret_cast<float4*>(St + qi * LDE + 4 * ty) = make_float4(s4[0], s4[1], s4[2], s4[3]);
    }
    __syncthreads();
#pragma unroll 2
    for (int ii = 0; ii < BT; ++ii) {
      const float4 p4 = *reinterpret_cast<const float4*>(Pt + ii * LDE + 4 * ty);
      const float4 s4 = *reinterpret_cast<const float4*>(St + ii * LDE + 4 * ty);
      float dov[DT], qv[DT];
#pragma unroll
      for (int x = 0; x < DT / 4; ++x) {
        const float4 w = *reinterpret_cast<const float4*>(Dt + ii * LDT + DT * tx + 4 * x);
        const float4 u = *reinterpret_cast<const float4*>(Qt + ii * LDT + DT * tx + 4 * x);
        dov[4 * x] = w.x;
        dov[4 * x + 1] = w.y;
        dov[4 * x + 2] = w.z;
        dov[4 * x + 3] = w.w;
        qv[4 * x] = u.x;
        qv[4 * x + 1] = u.y;
        qv[4 * x + 2] = u.z;
        qv[4 * x + 3] = u.w;
      }
      const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
      const float sr[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int d = 0; d < DT; ++d) {
          adv[r][d] = fmaf(pr[r], dov[d], adv[r][d]);
          adk[r][d] = fmaf(sr[r], qv[d], adk[r][d]);
        }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = j0 + 4 * ty + r;
    if (j >= s.NK) continue;
    const size_t ko = static_cast<size_t>(bh) * s.NK + j;
#pragma unroll
    for (int d = 0; d < DT; ++d) {
      store_val(dk, ko * D + DT * tx + d, s.scale * adk[r][d], grad_bf16);
      store_val(dv, ko * D + DT * tx + d, adv[r][d], grad_bf16);
    }
  }
}

template <int D>
cudaError_t fwd_simt_d(const AttnShape& s, const float* q, const float* k, const float* v, void* o, bool out_bf16,
                       float* row_m, float* row_s, int32_t* row_arg, cudaStream_t st) {
  if constexpr (D == 64 || D == 128) {
    using T = TiledGeom<D>;
    const cudaError_t e = cudaFuncSetAttribute(attn_fwd_simt_tiled_kernel<D>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((s.NQ + T::BQ - 1) / T::BQ, s.B * s.H);
    attn_fwd_simt_tiled_kernel<D><<<grid, T::THREADS, T::SMEM_BYTES, st>>>(s, q, k, v, o, out_bf16 ? 1 : 0, row_m,
                                                                           row_s, row_arg);
  } else {
    dim3 grid((s.NQ + SimtGeom<D>::ROWS - 1) / SimtGeom<D>::ROWS, s.B * s.H);
    attn_fwd_simt_kernel<D><<<grid, 128, 0, st>>>(s, q, k, v, o, out_bf16 ? 1 : 0, row_m, row_s, row_arg);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_simt_d(const AttnShape& s, const float* q, const float* k, const float* v, const void* o,
                       bool o_bf16, const float* dout, const float* row_m, const float* row_s,
                       const int32_t* row_arg, void* dq, void* dk, void* dv, bool grad_bf16, float* ws_d,
                       float* ws_r, cudaStream_t st) {
  if constexpr (D == 64 || D == 128) {
    using T = TiledBwdGeom<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_simt_tiled_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::DQ_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dkdv_simt_tiled_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T::KV_BYTES);
    if (e != cudaSuccess) return e;
    dim3 gq((s.NQ + T::BR - 1) / T::BR, s.B * s.H);
    attn_bwd_dq_simt_tiled_kernel<D><<<gq, T::THREADS, T::DQ_BYTES, st>>>(
        s, q, k, v, o, o_bf16 ? 1 : 0, dout, row_m, row_s, row_arg, dq, grad_bf16 ? 1 : 0, ws_d, ws_r);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 gk((s.NK + T::BR - 1) / T::BR, s.B * s.H);
    attn_bwd_dkdv_simt_tiled_kernel<D><<<gk, T::THREADS, T::KV_BYTES, st>>>(
        s, q, k, v, dout, row_m, row_s, row_arg, dk, dv, grad_bf16 ? 1 : 0, ws_d, ws_r);
    return cudaGetLastError();
  } else {
    dim3 gq((s.NQ + SimtGeom<D>::ROWS - 1) / SimtGeom<D>::ROWS, s.B * s.H);
    attn_bwd_dq_simt_kernel<D><<<gq, 128, 0, st>>>(s, q, k, v, o, o_bf16 ? 1 : 0, dout, row_m, row_s, row_arg,
                                                   dq, grad_bf16 ? 1 : 0, ws_d, ws_r);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 gk((s.NK + SimtGeom<D>::ROWS - 1) / SimtGeom<D>::ROWS, s.B * s.H);
    attn_bwd_dkdv_simt_kernel<D><<<gk, 128, 0, st>>>(s, q, k, v, dout, row_m, row_s, row_arg, dk, dv,
                                                     grad_bf16 ? 1 : 0, ws_d, ws_r);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_attn_fwd_simt(const AttnShape& s, const float* q, const float* k, const float* v, void* o,
                                 bool out_bf16, float* row_m, float* row_s, int32_t* row_arg, cudaStream_t st) {
  switch (s.D) {
    case 16: return fwd_simt_d<16>(s, q, k, v, o, out_bf16, row_m, row_s, row_arg, st);
    case 32: return fwd_simt_d<32>(s, q, k, v, o, out_bf16, row_m, row_s, row_arg, st);
    case 64: return fwd_simt_d<64>(s, q, k, v, o, out_bf16, row_m, row_s, row_arg, st);
    case 128: return fwd_simt_d<128>(s, q, k, v, o, out_bf16, row_m, row_s, row_arg, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_bwd_simt(const AttnShape& s, const float* q, const float* k, const float* v,
                                 const void* o, bool o_bf16, const float* dout, const float* row_m,
                                 const float* row_s, const int32_t* row_arg, void* dq, void* dk, void* dv,
                                 bool grad_bf16, float* ws_d, float* ws_r, cudaStream_t st) {
  switch (s.D) {
    case 16: return bwd_simt_d<16>(s, q, k, v, o, o_bf16, dout, row_m, row_s, row_arg, dq, dk, dv, grad_bf16, ws_d, ws_r, st);
    case 32: return bwd_simt_d<32>(s, q, k, v, o, o_bf16, dout, row_m, row_s, row_arg, dq, dk, dv, grad_bf16, ws_d, ws_r, st);
    case 64: return bwd_simt_d<64>(s, q, k, v, o, o_bf16, dout, row_m, row_s, row_arg, dq, dk, dv, grad_bf16, ws_d, ws_r, st);
    case 128: return bwd_simt_d<128>(s, q, k, v, o, o_bf16, dout, row_m, row_s, row_arg, dq, dk, dv, grad_bf16, ws_d, ws_r, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace raattn
