// w4_quant.cu — dynamic per-token int8 quantization of the activations that
// feed the W4A8 GEMM.  vLLM PR #6547 "Enable Dynamic Per Token fp8": one
// activation scale per token, computed at run time from that token's own
// values; pytorch/ao PR #1113 "support W4A8 Marlin kernel": the W4A8
// activations are symmetric int8.  For every row m of a [M,K]:
//
//   s_tok[m] = max_k |a[m][k]| / 127                (fp32, one rounding)
//   q[m][k]  = a[m][k] / s_tok[m] rounded once to fp32, then to the nearest
//              integer (ties to even); a row of zeros gets s_tok 0, codes 0.
//
// One CTA per row; the work is HBM-bound (2 bytes read and 1 written per
// element).  The first pass streams the row with 16-byte loads, four in
// flight per thread, and reduces |a| to the row maximum; the second pass
// reads the row again — from L2, where the first pass just left it — and
// writes eight codes per 8-byte store.  Rows whose length or addresses do
// not allow 16-byte loads take the same two passes one element at a time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int kQuantThreads = 256;

template <typename T>
__device__ __forceinline__ float2 pair_f32(uint32_t v);
template <>
__device__ __forceinline__ float2 pair_f32<__half>(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
template <>
__device__ __forceinline__ float2 pair_f32<__nv_bfloat16>(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}
template <typename T>
__device__ __forceinline__ float one_f32(T x);
template <>
__device__ __forceinline__ float one_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float one_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// Largest |x| of the eight 16-bit values in v.
template <typename T>
__device__ __forceinline__ float max8(const uint4& v) {
  const float2 a = pair_f32<T>(v.x), b = pair_f32<T>(v.y), c = pair_f32<T>(v.z),
               d = pair_f32<T>(v.w);
  const float m0 = fmaxf(fabsf(a.x), fabsf(a.y)), m1 = fmaxf(fabsf(b.x), fabsf(b.y));
  const float m2 = fmaxf(fabsf(c.x), fabsf(c.y)), m3 = fmaxf(fabsf(d.x), fabsf(d.y));
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// The int8 code of x as a byte: the correctly rounded fp32 quotient x / s,
// rounded to the nearest integer with ties to even.  |x| <= amax keeps the
// quotient within 127 * (1 + 2^-23); the clamp only guards that bound.
__device__ __forceinline__ uint32_t code(float x, float s) {
  float r = rintf(__fdiv_rn(x, s));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu;
}

// Eight codes of the 16-bit values in v, element j in byte j.
template <typename T>
__device__ __forceinline__ uint2 codes8(const uint4& v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float2 f = pair_f32<T>(w[p]);
    out[p >> 1] |= (code(f.x, s) | (code(f.y, s) << 8)) << (16 * (p & 1));
  }
  return make_uint2(out[0], out[1]);
}

template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
    quant_per_token_kernel(const T* __restrict__ a, int64_t K, int8_t* __restrict__ q,
                           float* __restrict__ s_tok, int vec) {
  __shared__ float red[kQuantThreads / 32];
  const int64_t m = blockIdx.x;
  const T* row = a + m * K;
  int8_t* qrow = q + m * K;

  // pass 1: the row maximum of |a|
  float amax = 0.f;
  if (vec) {
    const uint4* r8 = reinterpret_cast<const uint4*>(row);
    const int64_t n8 = K >> 3;
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < n8; i += kQuantThreads) amax = fmaxf(amax, max8<T>(__ldg(r8 + i)));
  } else {
    for (int64_t k = threadIdx.x; k < K; k += kQuantThreads) amax = fmaxf(amax, fabsf(one_f32(row[k])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, red[i]);

  const float s = __fdiv_rn(amax, 127.f);
  if (threadIdx.x == 0) s_tok[m] = s;
  const bool live = amax > 0.f;

  // pass 2: the codes
  if (vec) {
    const uint4* r8 = reinterpret_cast<const uint4*>(row);
    uint2* q8 = reinterpret_cast<uint2*>(qrow);
    const int64_t n8 = K >> 3;
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < n8; i += kQuantThreads)
      q8[i] = live ? codes8<T>(__ldg(r8 + i), s) : make_uint2(0u, 0u);
  } else {
    for (int64_t k = threadIdx.x; k < K; k += kQuantThreads)
      qrow[k] = static_cast<int8_t>(live ? code(one_f32(row[k]), s) : 0u);
  }
}

}  // namespace

cudaError_t launch_quant_per_token(bool bf16, const void* a, int64_t M, int64_t K, int8_t* q,
                                   float* s_tok, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int vec = K % 8 == 0 && reinterpret_cast<uintptr_t>(a) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(q) % 8 == 0;
  const dim3 grid(static_cast<unsigned>(M));
  if (bf16)
    quant_per_token_kernel<__nv_bfloat16><<<grid, kQuantThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a), K, q, s_tok, vec);
  else
    quant_per_token_kernel<__half><<<grid, kQuantThreads, 0, s>>>(static_cast<const __half*>(a),
                                                                   K, q, s_tok, vec);
  return cudaGetLastError();
}

}  // namespace w4
