// w4_dk.cu — the skinny-M ("decode") schedule of the 4-bit-weight GEMM:
// M <= 16 activation rows, HBM-bound on the weight bytes.
//
// Each warp owns 16 weight columns (n) of a 128-column tile and a range of
// 128-wide K blocks.  Per K block a thread loads two 16-byte chunks of the
// prepacked weights straight from global memory into registers (row g and
// row g+8 of its warp's 16 columns, chunk t of the block), turns each
// nibble pair into a 16-bit pair "magic + q" with one shift and one
// lop3 (exact), and feeds them as the A fragments of warp-level
// mma.sync.m16n8k16 (weights as the 16-row operand, activations as the
// 8-column operand).  The fp32 accumulator of one K block is then folded
// into the running result with the block's scale and zero-point:
//
//   sum_k a*w_hat = s*(sum_k a*(magic+q) - (magic+bias)*S) - w_z*S,
//   S = sum_k a over the block,
//
// which is exactly the per-element rule w_hat = (q - bias)*s - w_z of the
// Machete Readme ("Overview"), with the scale and pre-scaled zero-point
// applied once per block instead of once per weight.  For W4A8
// (pytorch/ao PR #1113 "support W4A8 Marlin kernel") the same identity is
// evaluated in int32: the block sums of int8 x (128+q) are integers below
// 2^24, exact in the fp32 accumulator, converted and corrected exactly.
//
// K order inside a block is permuted consistently for both operands: the
// MMA sums over K, so any consistent order gives the same products.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "w4_epilogue.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int kDkWarps = 8;          // 8 warps x 16 columns = one 128-column tile
constexpr int kDkThreads = 32 * kDkWarps;
constexpr int kBlockK = 128;         // K block: 4 chunks of 32
constexpr int kPrefetch = 4;         // K blocks of weights in flight per thread

// Position (0..31) inside a 32-wide chunk of the first K-value of pair p
// (0..15): word p/4 holds K 8*(p/4)..8*(p/4)+7 in ExLlama order, and its
// p%4-th nibble pair (bits 4*(p%4) and 16+4*(p%4)) is K 2*(p%4), 2*(p%4)+1.
__host__ __device__ __forceinline__ int pair_k(int p) { return 8 * (p >> 2) + 2 * (p & 3); }

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Four exact 16-bit pairs (magic + q) from one word; magic = 128 (bf16,
// 0x4300) or 1024 (f16, 0x6400).
template <bool F16>
__device__ __forceinline__ void word_pairs(uint32_t x, uint32_t (&o)[4]) {
  const uint32_t magic = F16 ? 0x64006400u : 0x43004300u;
  o[0] = lop_and_or(x, 0x000F000Fu, magic);
  o[1] = lop_and_or(x >> 4, 0x000F000Fu, magic);
  o[2] = lop_and_or(x >> 8, 0x000F000Fu, magic);
  o[3] = lop_and_or(x >> 12, 0x000F000Fu, magic);
}

template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace

// One CTA = one unit: 128 weight columns (tile nt) x K blocks [kb0, kb1).
// NJ = number of 8-row activation tiles (M <= 8 * NJ).
template <int MODE, int NJ>
__global__ void __launch_bounds__(kDkThreads, 2)
    dk_gemm_kernel(const void* __restrict__ act, const DkPlan p, const TcArgs args) {
  constexpr bool F16 = MODE == kW4A16_F16;
  using T16 = typename std::conditional<F16, __half, __nv_bfloat16>::type;
  extern __shared__ __align__(16) uint8_t smem[];
  const int64_t M = args.M, N = args.N, K = args.K;
  const int nt = blockIdx.x % p.n_tiles;
  const int split = blockIdx.x / p.n_tiles;
  const int kb0 = static_cast<int>(static_cast<int64_t>(split) * p.kblocks / p.ksplit);
  const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.kblocks / p.ksplit);
  const int nkb = kb1 - kb0;
  // shared memory: permuted activation fragments, then block row sums
  uint2* sact = reinterpret_cast<uint2*>(smem);                        // [nkb][8][NJ][32]
  float* ssum = reinterpret_cast<float*>(smem + static_cast<size_t>(p.kbu_max) * 8 * NJ * 32 * 8);
  int* isum = reinterpret_cast<int*>(ssum);                              // [nkb][8*NJ]

  // ---- weight stream: kPrefetch 128-wide K blocks of weights (and their
  // scale / zero rows) in flight per thread; the first loads are issued
  // before the activations are staged, so their latency overlaps staging.
  // Every per-load index advances incrementally (no multiplies, no
  // divisions in the loop).
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int ra = warp * 16 + g, rb = ra + 8;                  // rows within the tile
  const int64_t na = static_cast<int64_t>(nt) * kTileN + ra, nb = na + 8;
  const int64_t chunks = K / kChunkK;
  const int full_blocks = static_cast<int>(chunks >> 2);      // blocks with all 4 chunks
  const bool t_in_last = t < static_cast<int>(chunks & 3);    // chunk t of a partial last block
  const int kb_per_g = args.group_size >= K ? (1 << 30) : static_cast<int>(args.group_size / kBlockK);
  const bool pc = args.group_size >= K;                       // one group per column
  constexpr float kMagic = F16 ? 1024.f : 128.f;
  constexpr bool kSubMagic = F16;  // f16: subtract magic+bias exactly before the MMA
  const bool rowa_ok = na < N, rowb_ok = nb < N;
  const uint8_t* wptr = args.b_packed +
                        ((static_cast<int64_t>(nt) * chunks + static_cast<int64_t>(kb0) * 4 + t) *
                             kTileN + ra) * 16;
  constexpr int64_t kWStep = 4 * kTileN * 16;  // bytes from one K block to the next
  // scale / zero-point row pointers of the current group (column na; nb is +8)
  const int64_t g0 = pc ? 0 : kb0 / kb_per_g;
  const T16* scp = static_cast<const T16*>(args.scales) + g0 * N + na;
  const T16* zpp = static_cast<const T16*>(args.zeros) + g0 * N + na;
  const int8_t* sgp = static_cast<const int8_t*>(args.scales) + g0 * N + na;
  int gleft = pc ? (1 << 30) : kb_per_g - kb0 % kb_per_g;     // blocks left in this group
  int kb_next = kb0;

  auto rd_s = [&](float& va, float& vb, float& wz_a, float& wz_b) {
    if (MODE == kW4A8) {
      va = (args.scales && rowa_ok) ? static_cast<float>(sgp[0]) : 1.f;
      vb = (args.scales && rowb_ok) ? static_cast<float>(sgp[8]) : 1.f;
    } else {
      va = rowa_ok ? to_f32(scp[0]) : 0.f;
      vb = rowb_ok ? to_f32(scp[8]) : 0.f;
      wz_a = (args.zeros && rowa_ok) ? to_f32(zpp[0]) : 0.f;
      wz_b = (args.zeros && rowb_ok) ? to_f32(zpp[8]) : 0.f;
    }
  };
  // one group per column: the scale / zero rows never change
  float pc_sa = 1.f, pc_sb = 1.f, pc_za = 0.f, pc_zb = 0.f;
  if (pc) rd_s(pc_sa, pc_sb, pc_za, pc_zb);

  uint4 wa[kPrefetch], wb[kPrefetch];
  float sa[kPrefetch], sb[kPrefetch], za[kPrefetch], zb[kPrefetch];
  auto load = [&](int slot) {
    if (kb_next < full_blocks || (kb_next == full_blocks && t_in_last)) {
      wa[slot] = ldg_nc_v4(wptr);
      wb[slot] = ldg_nc_v4(wptr + 8 * 16);
    } else {
      wa[slot] = make_uint4(0, 0, 0, 0);
      wb[slot] = make_uint4(0, 0, 0, 0);
    }
    wptr += kWStep;
    ++kb_next;
    if (!pc) {
      rd_s(sa[slot], sb[slot], za[slot], zb[slot]);
      if (--gleft == 0) {
        gleft = kb_per_g;
        scp += N;
        zpp += N;
        sgp += N;
      }
    }
  };
#pragma unroll
  for (int q = 0; q < kPrefetch; ++q)
    if (q < nkb) load(q);

  // ---- stage this unit's activations, K-permuted to match the weight
  // fragments.  One task = 8 consecutive K values of one row (one prepacked
  // word's K range): a single 16-byte (8-byte for int8) load, scattered as
  // four 16-bit pairs.  Pair h of word w of chunk t is pair p = 4w + h of
  // the chunk, which MMA i = p / 2 uses as its b0 (p even) or b1 (p odd).
  {
    const int tasks = nkb * 16 * 8 * NJ;  // blocks x 16 words x rows
    for (int task = threadIdx.x; task < tasks; task += blockDim.x) {
      const int m = task % (8 * NJ);
      const int wg = (task / (8 * NJ)) % 16;  // word within the block: chunk wg/4, word wg%4
      const int kbl = task / (8 * NJ) / 16;
      const int tt = wg >> 2, w = wg & 3;
      const int64_t k0 = static_cast<int64_t>(kb0 + kbl) * kBlockK + 8 * wg;
      uint32_t pr[4] = {0u, 0u, 0u, 0u};
      if (m < M && k0 < K) {  // K % 64 == 0, so a word's 8 K values are all in or all out
        if (MODE == kW4A8) {
          const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const int8_t*>(act) + m * K + k0);
          const int8_t* b8 = reinterpret_cast<const int8_t*>(&raw);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            __nv_bfloat162 v = __floats2bfloat162_rn(static_cast<float>(b8[2 * h]),
                                                     static_cast<float>(b8[2 * h + 1]));
            pr[h] = *reinterpret_cast<uint32_t*>(&v);
          }
        } else {
          const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const T16*>(act) + m * K + k0);
          pr[0] = raw.x;
          pr[1] = raw.y;
          pr[2] = raw.z;
          pr[3] = raw.w;
        }
      }
      const int j = m >> 3, gg = m & 7;
      uint32_t* base32 = reinterpret_cast<uint32_t*>(sact);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int pp = 4 * w + h, i = pp >> 1;
        base32[((((kbl * 8 + i) * NJ + j) * 32) + gg * 4 + tt) * 2 + (pp & 1)] = pr[h];
      }
    }
  }
  __syncthreads();
  // block row sums S[kbl][m] over the staged values, fixed reduction order:
  // lane (i = lane/4, t = lane%4) adds the four values of its fragment entry
  {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int w = warp; w < nkb * 8 * NJ; w += kDkWarps) {
      const int kbl = w / (8 * NJ), m = w % (8 * NJ);
      const int j = m >> 3, gg = m & 7, i = lane >> 2, tt = lane & 3;
      const uint2 e = sact[((kbl * 8 + i) * NJ + j) * 32 + gg * 4 + tt];
      float v4[4];
      if constexpr (F16) {
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&e.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&e.y));
        v4[0] = f0.x; v4[1] = f0.y; v4[2] = f1.x; v4[3] = f1.y;
      } else {
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&e.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&e.y));
        v4[0] = f0.x; v4[1] = f0.y; v4[2] = f1.x; v4[3] = f1.y;
      }
      if (MODE == kW4A8) {
        int si = static_cast<int>(v4[0]) + static_cast<int>(v4[1]) + static_cast<int>(v4[2]) +
                 static_cast<int>(v4[3]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) si += __shfl_xor_sync(0xffffffffu, si, o);
        if (lane == 0) isum[kbl * 8 * NJ + m] = si;
      } else {
        float sf = (v4[0] + v4[1]) + (v4[2] + v4[3]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sf += __shfl_xor_sync(0xffffffffu, sf, o);
        if (lane == 0) ssum[kbl * 8 * NJ + m] = sf;
      }
    }
  }
  __syncthreads();

  float res[NJ][4];
  int32_t ires[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      res[j][e] = 0.f;
      ires[j][e] = 0;
    }

  const uint32_t off2 = kSubMagic ? [&] {
    __half2 h = __float2half2_rn(kMagic + static_cast<float>(args.wbias));
    return *reinterpret_cast<uint32_t*>(&h);
  }() : 0u;

  for (int kbl0 = 0; kbl0 < nkb; kbl0 += kPrefetch) {
#pragma unroll
    for (int q = 0; q < kPrefetch; ++q) {
      const int kbl = kbl0 + q;
      if (kbl >= nkb) break;
      // dequantize: pairs (magic + q) of rows a and b, 16 each
      uint32_t pa[16], pb[16];
      {
        const uint32_t xa[4] = {wa[q].x, wa[q].y, wa[q].z, wa[q].w};
        const uint32_t xb[4] = {wb[q].x, wb[q].y, wb[q].z, wb[q].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t o[4];
          word_pairs<F16>(xa[w], o);
#pragma unroll
          for (int h = 0; h < 4; ++h) pa[4 * w + h] = o[h];
          word_pairs<F16>(xb[w], o);
#pragma unroll
          for (int h = 0; h < 4; ++h) pb[4 * w + h] = o[h];
        }
        if constexpr (kSubMagic) {
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            __half2 va = __hsub2(*reinterpret_cast<__half2*>(&pa[h]), *reinterpret_cast<const __half2*>(&off2));
            __half2 vb = __hsub2(*reinterpret_cast<__half2*>(&pb[h]), *reinterpret_cast<const __half2*>(&off2));
            pa[h] = *reinterpret_cast<uint32_t*>(&va);
            pb[h] = *reinterpret_cast<uint32_t*>(&vb);
          }
        }
      }
      const float s_a = pc ? pc_sa : sa[q], s_b = pc ? pc_sb : sb[q];
      const float z_a = pc ? pc_za : za[q], z_b = pc ? pc_zb : zb[q];
      if (kbl + kPrefetch < nkb) load(q);
      float acc[NJ][4], acc2[NJ][4];  // two independent MMA chains (even / odd i)
#pragma unroll
      for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[j][e] = 0.f;
          acc2[j][e] = 0.f;
        }
      const uint2* bp = sact + static_cast<size_t>(kbl) * 8 * NJ * 32 + lane;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t afr[4] = {pa[2 * i], pb[2 * i], pa[2 * i + 1], pb[2 * i + 1]};
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const uint2 bv = bp[(i * NJ + j) * 32];
          mma16816<F16>((i & 1) ? acc2[j] : acc[j], afr, bv.x, bv.y);
        }
      }
#pragma unroll
      for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] += acc2[j][e];
      // fold the block into the running result
      if (MODE == kW4A8) {
        // block sums are integers below 2^22: adding 1.5*2^23 puts them in the
        // low mantissa bits, read back exactly as an int
        const int isa = static_cast<int>(s_a), isb = static_cast<int>(s_b);
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int2 S2 = *reinterpret_cast<const int2*>(&isum[kbl * 8 * NJ + j * 8 + 2 * t]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int bi = __float_as_int(acc[j][e] + 12582912.0f) - 0x4B400000;
            const int blk = bi - (128 + 8) * ((e & 1) ? S2.y : S2.x);
            if (pc) ires[j][e] += blk;
            else ires[j][e] += (e < 2 ? isa : isb) * blk;
          }
        }
      } else {
        const float mb = kMagic + static_cast<float>(args.wbias);
        const float c_a = kSubMagic ? z_a : fmaf(mb, s_a, z_a);
        const float c_b = kSubMagic ? z_b : fmaf(mb, s_b, z_b);
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const float2 S2 = *reinterpret_cast<const float2*>(&ssum[kbl * 8 * NJ + j * 8 + 2 * t]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float S = (e & 1) ? S2.y : S2.x;
            const float sr = e < 2 ? s_a : s_b, cr = e < 2 ? c_a : c_b;
            res[j][e] = fmaf(sr, acc[j][e], fmaf(-cr, S, res[j][e]));
          }
        }
      }
    }
  }

  // ---- epilogue: direct store, or split-K partials + last-arriver reduce
  auto store = [&](int64_t m, int64_t n, float vf, int32_t vi) {
    if (m >= M || n >= N) return;
    store_out<MODE>(args, m, n, vf, vi);
  };
  if (p.ksplit == 1) {
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        store(j * 8 + 2 * t + (e & 1), e < 2 ? na : nb, res[j][e], ires[j][e]);
    return;
  }
  const int MR = 8 * NJ;  // rows of a partial slot
  const size_t slot_elems = static_cast<size_t>(MR) * kTileN;
  float* pf = static_cast<float*>(args.partials);
  int32_t* pi = static_cast<int32_t*>(args.partials);
  const size_t my = (static_cast<size_t>(split) * p.n_tiles + nt) * slot_elems;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const size_t off = my + static_cast<size_t>(j * 8 + 2 * t + (e & 1)) * kTileN + (e < 2 ? ra : rb);
      if (MODE == kW4A8) pi[off] = ires[j][e];
      else pf[off] = res[j][e];
    }
  __threadfence();
  __syncthreads();
  __shared__ int last;
  if (threadIdx.x == 0) last = atomicAdd(&args.counters[nt], 1) == p.ksplit - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const size_t col = static_cast<size_t>(j * 8 + 2 * t + (e & 1)) * kTileN + (e < 2 ? ra : rb);
      float vf = 0.f;
      int32_t vi = 0;
      for (int sp = 0; sp < p.ksplit; ++sp) {
        const size_t off = (static_cast<size_t>(sp) * p.n_tiles + nt) * slot_elems + col;
        if (MODE == kW4A8) vi += __ldcg(pi + off);
        else vf = sp == 0 ? __ldcg(pf + off) : vf + __ldcg(pf + off);
      }
      store(j * 8 + 2 * t + (e & 1), e < 2 ? na : nb, vf, vi);
    }
  if (threadIdx.x == 0) args.counters[nt] = 0;  // leave the counter at zero for the next call
}

size_t dk_smem_bytes(int nj, int kbu_max) {
  return static_cast<size_t>(kbu_max) * 8 * nj * 32 * 8 + static_cast<size_t>(kbu_max) * 8 * nj * 4;
}

cudaError_t launch_dk(const DkPlan& plan, const void* a, const TcArgs& args, cudaStream_t s) {
  const void* fn = nullptr;
#define W4_DK_FN(MODE, NJ) reinterpret_cast<const void*>(&dk_gemm_kernel<MODE, NJ>)
  if (plan.mode == kW4A16_F16) fn = plan.nj == 1 ? W4_DK_FN(kW4A16_F16, 1) : W4_DK_FN(kW4A16_F16, 2);
  else if (plan.mode == kW4A16_BF16)
    fn = plan.nj == 1 ? W4_DK_FN(kW4A16_BF16, 1) : W4_DK_FN(kW4A16_BF16, 2);
  else fn = plan.nj == 1 ? W4_DK_FN(kW4A8, 1) : W4_DK_FN(kW4A8, 2);
#undef W4_DK_FN
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan.smem_bytes));
  if (e != cudaSuccess) return e;
  void* params[3] = {const_cast<void**>(&a), const_cast<DkPlan*>(&plan),
                     const_cast<TcArgs*>(&args)};
  return cudaLaunchKernel(fn, dim3(plan.grid), dim3(kDkThreads), params, plan.smem_bytes, s);
}

}  // namespace w4
