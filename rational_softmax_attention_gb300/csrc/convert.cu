// bf16 -> fp16 copies of attention operands, for the tensor-core products that take
// fp16 operands (P V in the forward; every product of the backward).
//
// A bf16 value has 8 significant bits and fp16 has 11, so the conversion is exact for
// |x| <= 65504 (values below 2^-14 become fp16 subnormals and keep at least their
// leading bits).  Larger magnitudes and NaN saturate and set kStatusRange in the
// library's status word.  HBM-bound: 2 bytes read and 2 written per element.
#include "kernels.cuh"

namespace raattn {
namespace {

// blockIdx.y selects the tensor; 8 values per 16-byte access, grid-stride.
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const ConvertJob job, unsigned int* status) {
  const int t = blockIdx.y;
  const uint4* __restrict__ src = job.src[t];
  uint4* __restrict__ dst = job.dst[t];
  const size_t n8 = job.n8[t];
  bool bad = false;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 u = __ldcs(src + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      bad |= !(fabsf(f.x) <= 65504.0f) || !(fabsf(f.y) <= 65504.0f);
      o[k] = pack_f16x2_sat(f.x, f.y);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusRange);
}

}  // namespace

cudaError_t launch_bf16_to_f16(const ConvertJob& job, unsigned int* status, cudaStream_t st) {
  if (job.count < 1 || job.count > 4) return cudaErrorInvalidValue;
  size_t nmax = 0;
  for (int i = 0; i < job.count; ++i) nmax = job.n8[i] > nmax ? job.n8[i] : nmax;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((nmax + 255) / 256, 152 * 8));
  bf16_to_f16_kernel<<<dim3(blocks > 0 ? blocks : 1, job.count), 256, 0, st>>>(job, status);
  return cudaGetLastError();
}

}  // namespace raattn
