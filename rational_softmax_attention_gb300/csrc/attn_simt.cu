// fp32 ra_attention on the CUDA cores (FFMA only, never TF32), forward and backward.
//
// Page "Ra-Family: Rational Neural Architecture", section 3, ra_attention
// (two passes per query tile: row maximum, then phi, sum(phi) and phi V) and
// ra_softmax "Closed-Form Backward Pass".  This path serves fp32 inputs, where
// the required accuracy (2e-5 absolute) rules out reduced-precision tensor cores.
//
// Layout of the work: a group of G = D/32 threads owns one query row (forward,
// dQ) or one key row (dK/dV); thread `part` of a group holds the dimensions
// d*G + part, so the G partial dot products are summed with G-1 xor shuffles.
// The other operand is staged in shared memory 32 rows at a time.  Scores are
// recomputed with exactly the same operation order in every kernel, so the
// argmax entry has Delta = 0 exactly in the second pass and in the backward.
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
  __shared__ float ks[KT][D];
  __shared__ float vs[KT][D];
  const int bh = blockIdx.y;
  const int r = threadIdx.x / G, part = threadIdx.x % G;
  const int i = blockIdx.x * ROWS + r;
  const bool row_ok = i < s.NQ;
  const float* qh = q + static_cast<size_t>(bh) * s.NQ * D;
  const float* kh = k + static_cast<size_t>(bh) * s.NK * D;
  const float* vh = v + static_cast<size_t>(bh) * s.NK * D;

  float qr[DPT];
#pragma unroll
  for (int d = 0; d < DPT; ++d) qr[d] = row_ok ? qh[static_cast<size_t>(i) * D + d * G + part] : 0.0f;
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
      float dot = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) dot = fmaf(qr[d], ks[jj][d * G + part], dot);
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
      float dot = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) dot = fmaf(qr[d], ks[jj][d * G + part], dot);
      dot = group_sum<G>(dot);
      const float sc = dot * s.scale;
      const int j = j0 + jj;
      const float delta = m - sc;
      if (j <= lim && delta < 16.0f) {
        const float phi = phi_exact(delta);
        sum += phi;
#pragma unroll
        for (int d = 0; d < DPT; ++d) acc[d] = fmaf(phi, vs[jj][d * G + part], acc[d]);
      }
    }
  }
  if (row_ok) {
    const size_t ro = static_cast<size_t>(bh) * s.NQ + i;
#pragma unroll
    for (int d = 0; d < DPT; ++d) store_val(o, ro * D + d * G + part, acc[d] / sum, out_bf16);
    if (part == 0) {
      if (row_m) row_m[ro] = m;
      if (row_s) row_s[ro] = sum;
      if (row_arg) row_arg[ro] = a;
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
  __shared__ float ks[KT][D];
  __shared__ float vs[KT][D];
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
    const size_t idx = ro * D + d * G + part;
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
      float dot = 0.0f, dp = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) {
        dot = fmaf(qr[d], ks[jj][d * G + part], dot);
        dp = fmaf(dor[d], vs[jj][d * G + part], dp);
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
        for (int d = 0; d < DPT; ++d) acc[d] = fmaf(e, ks[jj][d * G + part], acc[d]);
      }
    }
  }
  if (row_ok) {
#pragma unroll
    for (int d = 0; d < DPT; ++d) {
      const float ka = kh[static_cast<size_t>(a) * D + d * G + part];
      store_val(dq, ro * D + d * G + part, s.scale * fmaf(-R, ka, acc[d]), grad_bf16);
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
  __shared__ float qs[KT][D];
  __shared__ float dos[KT][D];
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
    kr[d] = k[ko * D + d * G + part];
    vr[d] = v[ko * D + d * G + part];
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
      float dot = 0.0f, dp = 0.0f;
#pragma unroll
      for (int d = 0; d < DPT; ++d) {
        dot = fmaf(qs[ii][d * G + part], kr[d], dot);
        dp = fmaf(dos[ii][d * G + part], vr[d], dp);
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
          adk[d] = fmaf(ds, qs[ii][d * G + part], adk[d]);
          adv[d] = fmaf(p, dos[ii][d * G + part], adv[d]);
        }
      }
    }
  }
  if (key_ok) {
#pragma unroll
    for (int d = 0; d < DPT; ++d) {
      store_val(dk, ko * D + d * G + part, s.scale * adk[d], grad_bf16);
      store_val(dv, ko * D + d * G + part, adv[d], grad_bf16);
    }
  }
}

template <int D>
cudaError_t fwd_simt_d(const AttnShape& s, const float* q, const float* k, const float* v, void* o, bool out_bf16,
                       float* row_m, float* row_s, int32_t* row_arg, cudaStream_t st) {
  dim3 grid((s.NQ + SimtGeom<D>::ROWS - 1) / SimtGeom<D>::ROWS, s.B * s.H);
  attn_fwd_simt_kernel<D><<<grid, 128, 0, st>>>(s, q, k, v, o, out_bf16 ? 1 : 0, row_m, row_s, row_arg);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_simt_d(const AttnShape& s, const float* q, const float* k, const float* v, const void* o,
                       bool o_bf16, const float* dout, const float* row_m, const float* row_s,
                       const int32_t* row_arg, void* dq, void* dk, void* dv, bool grad_bf16, float* ws_d,
                       float* ws_r, cudaStream_t st) {
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
