// ra_softmax row kernels: forward (HBM-bound, row held in registers) and the
// closed-form backward.
//
// Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax:
//   Delta_i = x_max - x_i, u_i = Delta_i/16, q_i = (1-u_i)/(1+u_i),
//   phi_i = q_i^8 for u_i < 1 and exactly 0 otherwise, p_i = phi_i / sum(phi);
//   backward from d phi/du = -16 phi/(1-u^2) with the gradient of x_max
//   routed to the (lowest-index) argmax.
//
// Arithmetic of phi on the FMA pipe: with w = (1+u)/2 = 0.5 + Delta/32,
// saturated to [0, 1] (so every u >= 1 lands on w = 1), q = 1/w - 1 and
// phi = ((q^2)^2)^2.  At w = 1 the reciprocal is 1 to within a few ulp, so
// |q| < 3e-7 and q^8 < 1e-52 rounds to exactly 0.0 in fp32: the compact
// support is exact without a separate select.
#include "kernels.cuh"

namespace raattn {

__device__ __forceinline__ float ra_phi_fast(float delta) {
  const float w = fma_sat(delta, 1.0f / 32.0f, 0.5f);
  const float q = rcp_approx(w) - 1.0f;
  const float q2 = q * q;
  const float q4 = q2 * q2;
  return q4 * q4;
}

template <int THREADS>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) r = fmaxf(r, red[w]);
  __syncthreads();
  return r;
}

template <int THREADS>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) r += red[w];
  __syncthreads();
  return r;
}

// One CTA per row; the row (cols <= THREADS*4*VPT, cols % 4 == 0, 16-byte aligned rows)
// is read once with 128-bit loads into registers, reduced, transformed and written
// once with 128-bit streaming stores.  x may equal y.
template <int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS) ra_softmax_fwd_vec_kernel(const float* x, float* y, int cols) {
  __shared__ float red[THREADS / 32];
  const size_t row = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + row * static_cast<size_t>(cols));
  float4* yr = reinterpret_cast<float4*>(y + row * static_cast<size_t>(cols));
  const int n4 = cols >> 2;
  float4 v[VPT];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < n4) {
      v[i] = __ldcs(xr + idx);
      m = max3f(m, fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w));
    }
  }
  m = block_max<THREADS>(m, red);
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < n4) {
      v[i].x = ra_phi_fast(m - v[i].x);
      v[i].y = ra_phi_fast(m - v[i].y);
      v[i].z = ra_phi_fast(m - v[i].z);
      v[i].w = ra_phi_fast(m - v[i].w);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
  }
  s = block_sum<THREADS>(s, red);
  const float inv = 1.0f / s;   // s >= 1: the maximum contributes phi = 1
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < n4) {
      float4 p;
      p.x = v[i].x * inv;
      p.y = v[i].y * inv;
      p.z = v[i].z * inv;
      p.w = v[i].w * inv;
      __stcs(yr + idx, p);
    }
  }
}

// Any cols, any alignment: three sweeps over the row in global memory.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) ra_softmax_fwd_generic_kernel(const float* x, float* y,
                                                                         int64_t cols) {
  __shared__ float red[THREADS / 32];
  const size_t row = blockIdx.x;
  const float* xr = x + row * static_cast<size_t>(cols);
  float* yr = y + row * static_cast<size_t>(cols);
  float m = -INFINITY;
  for (int64_t c = threadIdx.x; c < cols; c += THREADS) m = fmaxf(m, xr[c]);
  m = block_max<THREADS>(m, red);
  float s = 0.0f;
  for (int64_t c = threadIdx.x; c < cols; c += THREADS) s += ra_phi_fast(m - xr[c]);
  s = block_sum<THREADS>(s, red);
  const float inv = 1.0f / s;
  for (int64_t c = threadIdx.x; c < cols; c += THREADS) yr[c] = ra_phi_fast(m - xr[c]) * inv;
}

// Backward: dx_j = p_j (dy_j - D) / (1 - u_j^2) for j != a with u_j < 1, 0 for u_j >= 1,
// dx_a = -(sum of the others); D = sum_k p_k dy_k, a = lowest index of the row max of x.
// 1/(1-u^2) is written as 256 / ((16 - Delta)(16 + Delta)).
template <int THREADS>
__global__ void __launch_bounds__(THREADS) ra_softmax_bwd_kernel(const float* x, const float* p,
                                                                 const float* dy, float* dx, int64_t cols) {
  __shared__ float red[THREADS / 32];
  __shared__ long long red_idx[THREADS / 32];
  const size_t row = blockIdx.x;
  const size_t off = row * static_cast<size_t>(cols);
  const float* xr = x + off;
  const float* pr = p + off;
  const float* gr = dy + off;
  float* dr = dx + off;
  // row max and its lowest index
  float m = -INFINITY;
  long long a = -1;
  for (int64_t c = threadIdx.x; c < cols; c += THREADS) {
    const float xv = xr[c];
    if (xv > m) { m = xv; a = c; }
  }
  const float mall = block_max<THREADS>(m, red);
  long long cand = (m == mall) ? a : (long long)cols;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long other = __shfl_xor_sync(0xffffffffu, cand, o);
    cand = other < cand ? other : cand;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red_idx[warp] = cand;
  __syncthreads();
  long long amin = red_idx[0];
  for (int w = 1; w < THREADS / 32; ++w) amin = red_idx[w] < amin ? red_idx[w] : amin;
  __syncthreads();
  // D = sum p dy
  float d = 0.0f;
  for (int64_t c = threadIdx.x; c < cols; c += THREADS) d = fmaf(pr[c], gr[c], d);
  d = block_sum<THREADS>(d, red);
  // e_j and their sum (excluding the argmax)
  float rsum = 0.0f;
  for (int64_t c = threadIdx.x; c < cols; c += THREADS) {
    const float delta = mall - xr[c];
    float e = 0.0f;
    if (c != amin && delta < 16.0f) e = 256.0f * pr[c] * (gr[c] - d) / ((16.0f - delta) * (16.0f + delta));
    rsum += e;
    if (c != amin) dr[c] = e;
  }
  rsum = block_sum<THREADS>(rsum, red);
  if (threadIdx.x == 0 && amin >= 0 && amin < cols) dr[amin] = -rsum;
}

// ----------------------------------------------------------------------------
// launchers
// ----------------------------------------------------------------------------
template <int THREADS, int VPT>
static cudaError_t launch_vec(const float* x, float* y, int64_t rows, int cols, cudaStream_t st) {
  ra_softmax_fwd_vec_kernel<THREADS, VPT><<<static_cast<unsigned>(rows), THREADS, 0, st>>>(x, y, cols);
  return cudaGetLastError();
}

cudaError_t launch_ra_softmax_fwd_f32(const float* x, float* y, int64_t rows, int64_t cols, cudaStream_t st) {
  const bool vec_ok = (cols % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) &&
                      ((reinterpret_cast<uintptr_t>(y) & 15u) == 0);
  if (vec_ok && cols <= 256) return launch_vec<64, 1>(x, y, rows, static_cast<int>(cols), st);
  if (vec_ok && cols <= 1024) return launch_vec<256, 1>(x, y, rows, static_cast<int>(cols), st);
  if (vec_ok && cols <= 2048) return launch_vec<256, 2>(x, y, rows, static_cast<int>(cols), st);
  if (vec_ok && cols <= 4096) return launch_vec<256, 4>(x, y, rows, static_cast<int>(cols), st);
  if (vec_ok && cols <= 8192) return launch_vec<256, 8>(x, y, rows, static_cast<int>(cols), st);
  if (vec_ok && cols <= 16384) return launch_vec<512, 8>(x, y, rows, static_cast<int>(cols), st);
  ra_softmax_fwd_generic_kernel<256><<<static_cast<unsigned>(rows), 256, 0, st>>>(x, y, cols);
  return cudaGetLastError();
}

cudaError_t launch_ra_softmax_bwd_f32(const float* x, const float* p, const float* dy, float* dx, int64_t rows,
                                      int64_t cols, cudaStream_t st) {
  ra_softmax_bwd_kernel<256><<<static_cast<unsigned>(rows), 256, 0, st>>>(x, p, dy, dx, cols);
  return cudaGetLastError();
}

}  // namespace raattn
