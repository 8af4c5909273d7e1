// w4_kernels.cu — prepack / unprepack of the 4-bit weights, the int8 -> bf16
// activation conversion used by W4A8, and the CUDA-core ("simt") schedule
// of the GEMM, which runs any shape the API accepts.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "w4_epilogue.cuh"
#include "w4_internal.h"

namespace w4 {

// Bit position of K-value j (0..7) of a word in ExLlama order
// (vLLM API page "rdna_hybrid_w4a16", pack_int4_exllama_shuffle):
// even j at 0,4,8,12 and odd j at 16,20,24,28.
__device__ __forceinline__ int exl_bit(int j) { return ((j & 1) << 4) | ((j >> 1) << 2); }

// Reorder the eight nibbles of a sequential word (value j at bits 4j) into
// ExLlama order, and back.
__device__ __forceinline__ uint32_t seq_to_exl(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) r |= ((w >> (4 * j)) & 0xFu) << exl_bit(j);
  return r;
}
__device__ __forceinline__ uint32_t exl_to_seq(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) r |= ((w >> exl_bit(j)) & 0xFu) << (4 * j);
  return r;
}

// Offset of the prepacked word holding K-values k0..k0+7 (k0 % 8 == 0) of
// weight column n.
__device__ __forceinline__ int64_t packed_word_index(int64_t K, int64_t n, int64_t k0) {
  int64_t tile = n / kTileN, r = n % kTileN;
  int64_t chunk = k0 / kChunkK, j = (k0 % kChunkK) / 8;
  return ((tile * (K / kChunkK) + chunk) * kTileN + r) * 4 + j;
}

__device__ __forceinline__ int64_t input_word_index(int layout, int64_t K, int64_t N, int64_t n,
                                                    int64_t k0) {
  return layout == 0 ? (k0 / 8) * N + n : n * (K / 8) + k0 / 8;
}

// One thread per prepacked word.  Rows n >= N (tile padding) get zero.
__global__ void prepack_kernel(const int32_t* __restrict__ w_q, int wtype, int layout, int64_t K,
                               int64_t N, uint32_t* __restrict__ out, int64_t total) {
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int64_t j = idx % 4, r = (idx / 4) % kTileN;
    int64_t chunk = (idx / (4 * kTileN)) % (K / kChunkK);
    int64_t tile = idx / (4 * kTileN * (K / kChunkK));
    int64_t n = tile * kTileN + r, k0 = chunk * kChunkK + j * 8;
    uint32_t word = 0;
    if (n < N) {
      uint32_t in = static_cast<uint32_t>(w_q[input_word_index(layout, K, N, n, k0)]);
      word = layout == 2 ? in : seq_to_exl(in);
      if (wtype == 2) word ^= 0x88888888u;  // int4 -> offset binary (value q' - 8)
    }
    out[idx] = word;
  }
}

// One thread per word of the requested layout.
__global__ void unprepack_kernel(const uint32_t* __restrict__ packed, int wtype, int layout,
                                 int64_t K, int64_t N, int32_t* __restrict__ w_q,
                                 int64_t total) {
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int64_t n, k0;
    if (layout == 0) {
      n = idx % N;
      k0 = (idx / N) * 8;
    } else {
      n = idx / (K / 8);
      k0 = (idx % (K / 8)) * 8;
    }
    uint32_t word = packed[packed_word_index(K, n, k0)];
    if (wtype == 2) word ^= 0x88888888u;
    w_q[idx] = static_cast<int32_t>(layout == 2 ? word : exl_to_seq(word));
  }
}

// int8 -> the bf16 value, four codes of a word at a time without the
// conversion unit: byte k of w ^ 0x80808080 is v + 128; placed in the low
// mantissa byte of 2^23 (the bit pattern 0x4B0000uu) it reads 2^23 + v + 128,
// so subtracting 2^23 + 128 leaves v exactly, and a pair of such floats
// rounds to bf16 exactly (|v| <= 128).
__device__ __forceinline__ void s8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  float f[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t bits;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(bits) : "r"(u), "r"(0x4B000000u), "r"(0x7540u | k));
    f[k] = __fsub_rn(__uint_as_float(bits), 8388736.f);  // 2^23 + 128
  }
  __nv_bfloat162 p0 = __floats2bfloat162_rn(f[0], f[1]);
  __nv_bfloat162 p1 = __floats2bfloat162_rn(f[2], f[3]);
  lo = *reinterpret_cast<uint32_t*>(&p0);
  hi = *reinterpret_cast<uint32_t*>(&p1);
}

// int8 activations -> the bf16 copy the tensor-core W4A8 schedule reads:
// sixteen codes (one 16-byte load, two 16-byte stores) per thread and
// step; an odd last group of eight goes by itself.
__global__ void a8_to_bf16_kernel(const int8_t* __restrict__ a, int64_t count8,
                                  uint4* __restrict__ out) {
  // the W4A8 tensor-core GEMM that follows may launch now: it streams weights
  // until this grid is complete
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t count16 = count8 >> 1;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count16;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(a)[i];
    uint4 o0, o1;
    s8x4_to_bf16x4(v.x, o0.x, o0.y);
    s8x4_to_bf16x4(v.y, o0.z, o0.w);
    s8x4_to_bf16x4(v.z, o1.x, o1.y);
    s8x4_to_bf16x4(v.w, o1.z, o1.w);
    out[2 * i] = o0;
    out[2 * i + 1] = o1;
  }
  if ((count8 & 1) && blockIdx.x == 0 && threadIdx.x == 0) {
    const uint2 v = reinterpret_cast<const uint2*>(a)[count8 - 1];
    uint4 o;
    s8x4_to_bf16x4(v.x, o.x, o.y);
    s8x4_to_bf16x4(v.y, o.z, o.w);
    out[count8 - 1] = o;
  }
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// CUDA-core W4A16: one thread per output, w_hat = fma(v, s, -w_z) rounded
// once to T, fp32 accumulation over k ascending.
template <typename T>
__global__ void simt_w4a16_kernel(const T* __restrict__ a, TcArgs args) {
  const int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (n >= args.N) return;
  const T* s = static_cast<const T*>(args.scales);
  const T* z = static_cast<const T*>(args.zeros);
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(args.b_packed);
  const int64_t K = args.K, N = args.N;
  for (int64_t m = blockIdx.y; m < args.M; m += gridDim.y) {
    float acc = 0.f;
    for (int64_t k0 = 0; k0 < K; k0 += 8) {
      uint32_t word = wp[packed_word_index(K, n, k0)];
      int64_t g = k0 / args.group_size;
      T sc = s[g * N + n];
      T zn = z ? T(-to_f(z[g * N + n])) : from_f<T>(0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int v = static_cast<int>((word >> exl_bit(j)) & 0xFu) - args.wbias;
        T w = __hfma(from_f<T>(static_cast<float>(v)), sc, zn);
        acc = fmaf(to_f(a[m * K + k0 + j]), to_f(w), acc);
      }
    }
    store_out<std::is_same<T, __half>::value ? kW4A16_F16 : kW4A16_BF16>(args, m, n, acc, 0);
  }
}

// CUDA-core W4A8: exact int32 accumulation of a * v * sg.
__global__ void simt_w4a8_kernel(const int8_t* __restrict__ a, TcArgs args) {
  const int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (n >= args.N) return;
  const int8_t* sg = static_cast<const int8_t*>(args.scales);
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(args.b_packed);
  const int64_t K = args.K, N = args.N;
  for (int64_t m = blockIdx.y; m < args.M; m += gridDim.y) {
    int32_t acc = 0;
    for (int64_t k0 = 0; k0 < K; k0 += 8) {
      uint32_t word = wp[packed_word_index(K, n, k0)];
      int32_t mul = sg ? static_cast<int32_t>(sg[(k0 / args.group_size) * N + n]) : 1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int32_t v = static_cast<int32_t>((word >> exl_bit(j)) & 0xFu) - 8;
        acc += static_cast<int32_t>(a[m * K + k0 + j]) * v * mul;
      }
    }
    store_out<kW4A8>(args, m, n, 0.f, acc);
  }
}

// CUDA-core W4A8 with E4M3 activations: fp32 accumulation, k ascending, of
// the exact products decode(a) * v.
__global__ void simt_w4a8f8_kernel(const __nv_fp8_storage_t* __restrict__ a, TcArgs args) {
  const int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (n >= args.N) return;
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(args.b_packed);
  const int64_t K = args.K;
  for (int64_t m = blockIdx.y; m < args.M; m += gridDim.y) {
    float acc = 0.f;
    for (int64_t k0 = 0; k0 < K; k0 += 8) {
      uint32_t word = wp[packed_word_index(K, n, k0)];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float v = static_cast<float>(static_cast<int>((word >> exl_bit(j)) & 0xFu) - 8);
        const __half h = __half(__nv_cvt_fp8_to_halfraw(a[m * K + k0 + j], __NV_E4M3));
        acc = fmaf(__half2float(h), v, acc);
      }
    }
    store_out<kW4A8F8>(args, m, n, acc, 0);
  }
}

static int grid_for(int64_t total, int threads) {
  int64_t b = (total + threads - 1) / threads;
  if (b > (1 << 20)) b = 1 << 20;
  return b < 1 ? 1 : static_cast<int>(b);
}

cudaError_t launch_prepack(const int32_t* w_q, int wtype, int layout, int64_t K, int64_t N,
                           uint8_t* out, cudaStream_t s) {
  int64_t n_pad = (N + kTileN - 1) / kTileN * kTileN;
  int64_t total = n_pad * (K / 8);
  prepack_kernel<<<grid_for(total, 256), 256, 0, s>>>(w_q, wtype, layout, K, N,
                                                     reinterpret_cast<uint32_t*>(out), total);
  return cudaGetLastError();
}

cudaError_t launch_unprepack(const uint8_t* packed, int wtype, int layout, int64_t K, int64_t N,
                             int32_t* w_q, cudaStream_t s) {
  int64_t total = N * (K / 8);
  unprepack_kernel<<<grid_for(total, 256), 256, 0, s>>>(
      reinterpret_cast<const uint32_t*>(packed), wtype, layout, K, N, w_q, total);
  return cudaGetLastError();
}

cudaError_t launch_a8_to_bf16(const int8_t* a, int64_t count, void* out, cudaStream_t s) {
  int64_t c8 = count / 8;
  a8_to_bf16_kernel<<<grid_for((c8 + 1) / 2, 256), 256, 0, s>>>(a, c8, static_cast<uint4*>(out));
  return cudaGetLastError();
}

// K == 0 with a bias: every output element is its column's bias (a product
// over no K values is zero), rounded to the output type.
__global__ void bias_rows_kernel(int64_t M, int64_t N, const uint16_t* __restrict__ bias,
                                 uint16_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < M * N;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = bias[i % N];
}

cudaError_t launch_bias_rows(int mode, int64_t M, int64_t N, const void* bias, bool w4a8,
                             void* out, cudaStream_t s) {
  (void)mode;
  (void)w4a8;  // 0 * s_tok * s_ch + bias rounds to bias: the output type is the bias type
  bias_rows_kernel<<<grid_for(M * N, 256), 256, 0, s>>>(
      M, N, static_cast<const uint16_t*>(bias), static_cast<uint16_t*>(out));
  return cudaGetLastError();
}

cudaError_t launch_simt(int mode, const void* a, const TcArgs& args, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((args.N + 127) / 128),
            static_cast<unsigned>(args.M < 65535 ? args.M : 65535));
  if (mode == kW4A16_F16)
    simt_w4a16_kernel<__half><<<grid, 128, 0, s>>>(static_cast<const __half*>(a), args);
  else if (mode == kW4A16_BF16)
    simt_w4a16_kernel<__nv_bfloat16>
        <<<grid, 128, 0, s>>>(static_cast<const __nv_bfloat16*>(a), args);
  else if (mode == kW4A8F8)
    simt_w4a8f8_kernel<<<grid, 128, 0, s>>>(static_cast<const __nv_fp8_storage_t*>(a), args);
  else
    simt_w4a8_kernel<<<grid, 128, 0, s>>>(static_cast<const int8_t*>(a), args);
  return cudaGetLastError();
}

}  // namespace w4
