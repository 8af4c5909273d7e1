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
// element).  The first pass streams the row with 16-byte loads and reduces
// |a| to the row maximum; the second pass reads the row again — from L2,
// where the first pass just left it, so DRAM sees it once — and writes eight
// codes per store.  Rows whose length or addresses do not allow 16-byte
// loads take the same two passes one element at a time.
//
// The same kernels make E4M3 codes for fp8 activations (vLLM PR #9855:
// W4A8 "including fp8 activations"): s_tok = amax / 448 and each code the
// E4M3 value nearest to fl32(a / s_tok), ties to even, saturated at 448.
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

// Running maximum of |x| over pairs of 16-bit values, kept packed: the
// maximum is exact in the input type, so it is taken there (one instruction
// per pair) and converted to fp32 once per thread.
template <typename T>
struct Pair16;
template <>
struct Pair16<__half> {
  using P = __half2;
  static __device__ __forceinline__ P zero() { return __float2half2_rn(0.f); }
  static __device__ __forceinline__ P amax(P m, uint32_t v) {
    return __hmax2(m, __habs2(*reinterpret_cast<const __half2*>(&v)));
  }
  static __device__ __forceinline__ float to_f32(P m) {
    return fmaxf(__low2float(m), __high2float(m));
  }
};
template <>
struct Pair16<__nv_bfloat16> {
  using P = __nv_bfloat162;
  static __device__ __forceinline__ P zero() { return __float2bfloat162_rn(0.f); }
  static __device__ __forceinline__ P amax(P m, uint32_t v) {
    return __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&v)));
  }
  static __device__ __forceinline__ float to_f32(P m) {
    return fmaxf(__low2float(m), __high2float(m));
  }
};
template <typename T>
__device__ __forceinline__ typename Pair16<T>::P amax8(typename Pair16<T>::P m, const uint4& v) {
  m = Pair16<T>::amax(m, v.x);
  m = Pair16<T>::amax(m, v.y);
  m = Pair16<T>::amax(m, v.z);
  return Pair16<T>::amax(m, v.w);
}

// ---------------------------------------------------------------------------
// Codes of all three kinds (int8, int8 as bf16 values — the operand the
// tensor-core W4A8 schedule reads — and E4M3) from the same two passes: the
// row maximum, then the codes from a second read of the row (from L2, where
// the first pass left it).
//
// int8 codes without a division per element: with r = 1/s rounded once to
// fp32, the product p = fl(x * r) differs from fl(x / s) by at most
// |x / s| * (2^-23 + 2^-24 + 2^-47) < 2.3e-5 for |x / s| <= 127 + 2^-16; so
// when p is farther than 2^-15 from every half-integer, both round to the
// same integer (ties to even only matter exactly at a half-integer), and
// only the few quotients that close are divided exactly.  (s below 2^-128
// makes r infinite: then every code takes the division.)
enum QuantOut { kOutS8 = 0, kOutBf16 = 1, kOutE4M3 = 2 };

// fast: r = 1/s is finite (s below 2^-128 takes the division everywhere)
__device__ __forceinline__ float code_s8_fast(float x, float s, float r, bool fast) {
  const float p = x * r;
  const float d = fabsf(p - truncf(p));  // distance above the integer toward zero
  float q = (!fast || fabsf(d - 0.5f) <= 0x1p-15f) ? rintf(__fdiv_rn(x, s)) : rintf(p);
  return fminf(fmaxf(q, -127.f), 127.f);
}

// The eight int8 codes of f[] (|f| <= amax, so every code is within
// [-127, 127]), rounded to nearest even, as t[e] = code + 1.5 * 2^23: adding
// that constant to a value of magnitude below 2^22 rounds it to an integer
// (nearest even, the FADD's own rounding) held in the low mantissa bits, so
// the low byte of t's bit pattern is the two's-complement code and t - 1.5 *
// 2^23 its exact value.  Codes come from the products p with r; a product
// whose distance to the nearest integer is 0.5 - 2^-15 or more (within
// 2^-15 of a half-integer), or any product when r is not finite, is replaced
// by the code of the exact quotient, in a branch taken for few vectors.
constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23
__device__ __forceinline__ void codes8_s8(const float (&f)[8], float s, float r, bool fast,
                                          float (&t)[8]) {
  // explicitly rounded operations: none may be fused or reassociated
  float dmax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float p = __fmul_rn(f[e], r);
    t[e] = __fadd_rn(p, kRoundMagic);
    dmax = fmaxf(dmax, fabsf(__fsub_rn(p, __fsub_rn(t[e], kRoundMagic))));
  }
  if (!fast || dmax >= 0.5f - 0x1p-15f) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float p = __fmul_rn(f[e], r);
      if (!fast || fabsf(__fsub_rn(p, __fsub_rn(t[e], kRoundMagic))) >= 0.5f - 0x1p-15f)
        t[e] = __fadd_rn(__fdiv_rn(f[e], s), kRoundMagic);
    }
  }
}

// Low bytes of four ints, in order, in one word.
__device__ __forceinline__ uint32_t pack4_s8(int a, int b, int c, int d) {
  uint32_t lo, hi, r;
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(lo) : "r"(a), "r"(b));
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(hi) : "r"(c), "r"(d));
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r) : "r"(lo), "r"(hi));
  return r;
}

// E4M3 byte of the correctly rounded quotient x / s: nearest-even,
// saturated at 448
__device__ __forceinline__ uint32_t code_e4m3(float x, float s) {
  uint16_t e2;
  const float v = __fdiv_rn(x, s);
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(e2) : "f"(0.f), "f"(v));
  return e2 & 0xFFu;
}

template <typename T, int OUT>
__global__ void __launch_bounds__(kQuantThreads)
    quant2_kernel(const T* __restrict__ a, int64_t K, void* __restrict__ q,
                  float* __restrict__ s_tok, int vec) {
  // a GEMM launched after this one may start its weight stream now: it reads
  // the codes and scales only after this grid is complete
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float red[kQuantThreads / 32];
  const int64_t m = blockIdx.x;
  const T* row = a + m * K;

  // pass 1: the row maximum of |a|
  float amax = 0.f;
  if (vec) {
    const uint4* r8 = reinterpret_cast<const uint4*>(row);
    const int64_t n8 = K >> 3;
    typename Pair16<T>::P m2 = Pair16<T>::zero();
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < n8; i += kQuantThreads) m2 = amax8<T>(m2, __ldg(r8 + i));
    amax = Pair16<T>::to_f32(m2);
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

  const float s = __fdiv_rn(amax, OUT == kOutE4M3 ? 448.f : 127.f);
  if (threadIdx.x == 0) s_tok[m] = s;
  const bool live = amax > 0.f;
  const float r = __frcp_rn(s);
  const bool fast = isfinite(r);

  // pass 2: the codes
  if (vec) {
    const uint4* r8 = reinterpret_cast<const uint4*>(row);
    const int64_t n8 = K >> 3;
#pragma unroll 2
    for (int64_t i = threadIdx.x; i < n8; i += kQuantThreads) {
      const uint4 v = __ldg(r8 + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float f[8];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float2 fp = pair_f32<T>(w[pp]);
        f[2 * pp] = fp.x;
        f[2 * pp + 1] = fp.y;
      }
      if constexpr (OUT == kOutE4M3) {
        uint32_t o[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          o[e >> 2] |= (live ? code_e4m3(f[e], s) : 0u) << (8 * (e & 3));
        reinterpret_cast<uint2*>(static_cast<uint8_t*>(q) + m * K)[i] = make_uint2(o[0], o[1]);
      } else {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = kRoundMagic;  // code 0
        if (live) codes8_s8(f, s, r, fast, t);
        if constexpr (OUT == kOutBf16) {
          uint32_t o[4];
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fsub_rn(t[2 * pp], kRoundMagic),
                                                            __fsub_rn(t[2 * pp + 1], kRoundMagic));
            o[pp] = *reinterpret_cast<const uint32_t*>(&b2);  // exact
          }
          reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(q) + m * K)[i] =
              make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          reinterpret_cast<uint2*>(static_cast<int8_t*>(q) + m * K)[i] = make_uint2(
              pack4_s8(__float_as_int(t[0]), __float_as_int(t[1]), __float_as_int(t[2]),
                       __float_as_int(t[3])),
              pack4_s8(__float_as_int(t[4]), __float_as_int(t[5]), __float_as_int(t[6]),
                       __float_as_int(t[7])));
        }
      }
    }
  } else {
    for (int64_t k = threadIdx.x; k < K; k += kQuantThreads) {
      const float x = one_f32(row[k]);
      if constexpr (OUT == kOutE4M3) {
        static_cast<uint8_t*>(q)[m * K + k] = static_cast<uint8_t>(live ? code_e4m3(x, s) : 0u);
      } else {
        const float c = live ? code_s8_fast(x, s, r, fast) : 0.f;
        if constexpr (OUT == kOutBf16)
          static_cast<__nv_bfloat16*>(q)[m * K + k] = __float2bfloat16_rn(c);
        else
          static_cast<int8_t*>(q)[m * K + k] = static_cast<int8_t>(static_cast<int>(c));
      }
    }
  }
}

template <typename T>
cudaError_t launch_quant_t(int out, const void* a, int64_t M, int64_t K, void* q, float* s_tok,
                           cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(M));
  const int vec = K % 8 == 0 && reinterpret_cast<uintptr_t>(a) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(q) % (out == kOutBf16 ? 16 : 8) == 0;
  const T* at = static_cast<const T*>(a);
  if (out == kOutS8) quant2_kernel<T, kOutS8><<<grid, kQuantThreads, 0, s>>>(at, K, q, s_tok, vec);
  else if (out == kOutBf16)
    quant2_kernel<T, kOutBf16><<<grid, kQuantThreads, 0, s>>>(at, K, q, s_tok, vec);
  else quant2_kernel<T, kOutE4M3><<<grid, kQuantThreads, 0, s>>>(at, K, q, s_tok, vec);
  return cudaGetLastError();
}

}  // namespace

// out: 0 int8 codes, 1 int8 codes stored as bf16 values, 2 E4M3 codes
cudaError_t launch_quant_per_token(bool bf16, const void* a, int64_t M, int64_t K, void* q,
                                   float* s_tok, int out, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  return bf16 ? launch_quant_t<__nv_bfloat16>(out, a, M, K, q, s_tok, s)
              : launch_quant_t<__half>(out, a, M, K, q, s_tok, s);
}

}  // namespace w4
