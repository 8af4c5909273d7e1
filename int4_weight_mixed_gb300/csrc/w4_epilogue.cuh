#pragma once
// w4_epilogue.cuh — the output step shared by every GEMM engine.
//
//   W4A16: out[m][n] = round_T(sum + bias[n])            (T = fp16 / bf16)
//   W4A8 : out[m][n] = fp16_rn((float)acc * s_tok[m] * s_ch[n] + bias[n])
//          or the raw int32 accumulator (no scales, no bias); with fp8
//          activations acc is the fp32 sum of the exact products
//
// The sum is the fp32 (W4A16) or exact int32 (W4A8) result of the product;
// the products by the per-token and per-channel scales are taken left to
// right in fp32 (vLLM PR #6547 "Enable Dynamic Per Token fp8": per-token x
// per-channel scales applied in the epilogue); the optional bias [N], of the
// output type, is added in fp32 before the single rounding to the output
// type (the vLLM "rdna_hybrid_w4a16" page adds the layer bias to the GEMM
// result, _rdna_hybrid_w4a16_apply_impl).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "w4_internal.h"

namespace w4 {

template <typename T>
__device__ __forceinline__ float ep_f32(T x);
template <>
__device__ __forceinline__ float ep_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float ep_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T ep_round(float x);
template <>
__device__ __forceinline__ __half ep_round<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 ep_round<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Store output element (m, n) (both in range): vf is the fp32 sum (W4A16),
// vi the int32 accumulator (W4A8).
template <int MODE>
__device__ __forceinline__ void store_out(const TcArgs& args, int64_t m, int64_t n, float vf,
                                          int32_t vi) {
  const int64_t o = m * args.N + n;
  if constexpr (MODE == kW4A8F8) {  // fp32 sum of the exact E4M3 x int4 products
    float r = vf * args.s_tok[m] * args.s_ch[n];
    if (args.bias) r += ep_f32(static_cast<const __half*>(args.bias)[n]);
    static_cast<__half*>(args.out)[o] = __float2half_rn(r);
  } else if constexpr (MODE == kW4A8) {
    if (args.out_s32) {
      static_cast<int32_t*>(args.out)[o] = vi;
      return;
    }
    float r = static_cast<float>(vi) * args.s_tok[m] * args.s_ch[n];
    if (args.bias) r += ep_f32(static_cast<const __half*>(args.bias)[n]);
    static_cast<__half*>(args.out)[o] = __float2half_rn(r);
  } else {
    using T16 = typename std::conditional<MODE == kW4A16_F16, __half, __nv_bfloat16>::type;
    if (args.bias) vf += ep_f32(static_cast<const T16*>(args.bias)[n]);
    static_cast<T16*>(args.out)[o] = ep_round<T16>(vf);
  }
}

}  // namespace w4
