// w4_ds.cu — the streamed skinny-M ("decode") schedule of the 4-bit-weight
// GEMM: M <= 16 activation rows, HBM-bound on the weight bytes.
//
// Two kernels, the second launched as a programmatic dependent of the first
// so that its weight stream starts while the first still runs:
//
//   ds_prep   : rearranges the activations of every 128-wide K block into
//               the register order of the mma.sync B fragments ("frag"),
//               int8 -> bf16 for W4A8 (exact), and writes the block row sums
//               S[kb][m] that fold the dequantization offset out of the MMA.
//   ds_gemm   : persistent CTAs, two per SM, over a stream-K split of the
//               (weight tile, K block) iterations.  One producer thread
//               streams the prepacked nibbles of each two-block stage (one
//               contiguous bulk copy: a 128-column tile keeps its K range in
//               one run) and the stage's scale / zero-point rows; a second one
//               streams the matching activation fragments and row sums (one
//               copy) once the prep kernel is complete.  Four consumer warps
//               own 32 weight columns each: ldmatrix
//               hands every thread word t of its rows' four 32-K chunks, each
//               nibble pair becomes the 16-bit pair (magic + q) with one
//               shift and one lop3 (exact), and warp-level mma.sync.m16n8k16
//               accumulates a K block in fp32.  The block is folded into the
//               running result with its scale and zero-point:
//
//                 sum_k a*w_hat = s*(sum_k a*(magic+q) - (magic+bias)*S) - w_z*S
//
//               which is the per-element rule w_hat = (q - bias)*s - w_z of
//               the Machete Readme ("Overview"), applied once per block.
//               W4A8 (pytorch/ao PR #1113 "support W4A8 Marlin kernel") does
//               the same in int32: block sums of int8 x (128+q) stay below
//               2^22, exact in fp32, then converted and corrected exactly.
//
// K order inside a 128-K block: thread t of an MMA quad holds word t of each
// 32-K chunk c, i.e. K = 32c + 8t + 0..7; MMA i = 2c + h uses the pairs
// 2h, 2h+1 of that word (K 32c + 8t + 4h + 0..3).  The activation fragments
// are staged in exactly that order, so both operands agree on every K.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdio>
#include <cstdlib>

#include "w4_epilogue.cuh"
#include "w4_internal.h"
#include "w4_ptx.cuh"

namespace w4 {
namespace {

// A consumer warp owns kDsRP pairs of 8-row groups (16 weight columns per
// pair, one m16n8k16 A tile).  Two or three CTAs of six warps share an SM;
// the register file is split between the four SM sub-partitions, so their
// warps sit three deep (at most 168 registers a thread) or five deep (at
// most 96) per sub-partition.
// Up to 16 rows: 32 weight columns per warp (four consumer warps); 32 rows:
// 16 columns per warp (eight consumer warps), so that the accumulators of
// four activation tiles fit in registers.
template <int NJ>
struct DsShape {
  static constexpr int RP = NJ >= 4 ? 1 : 2;
  static constexpr int Cols = 16 * RP;
  static constexpr int Consumers = kTileN / Cols;
  static constexpr int WProd = Consumers;      // weight producer warp
  static constexpr int AProd = Consumers + 1;  // activation producer warp
  static constexpr int Threads = 32 * (Consumers + 2);
};
constexpr int kDsSB = 2;                          // K blocks per pipeline stage
constexpr int kBlkK = 128;
constexpr uint32_t kWBlk = 4 * kTileN * 16;       // prepacked bytes of one K block of a tile

struct DsUnit {
  int tile;
  int kb0, kb1;   // K blocks of this tile handled by this CTA
  int nslots;     // CTAs contributing to the tile
  int cfirst;     // first of them
  int seg;        // index of this tile among the CTA's tiles
};

__device__ __forceinline__ int64_t ds_start(int64_t c, int64_t T, int64_t G) { return div_nn(c * T, G); }
__device__ __forceinline__ int64_t ds_owner(int64_t i, int64_t T, int64_t G) {
  return div_nn((i + 1) * G - 1, T);
}

// u-th tile segment of this CTA's stream-K range; false when there is none.
__device__ __forceinline__ bool ds_unit(const DsPlan& p, int u, DsUnit& o) {
  const int64_t T = static_cast<int64_t>(p.n_tiles) * p.kblocks, G = p.grid;
  const int64_t b = ds_start(blockIdx.x, T, G), e = ds_start(blockIdx.x + 1, T, G);
  if (b >= e) return false;
  const int64_t t = div_nn(b, p.kblocks) + u;
  int64_t lo = t * p.kblocks, hi = lo + p.kblocks;
  if (lo < b) lo = b;
  if (hi > e) hi = e;
  if (lo >= hi) return false;
  o.tile = static_cast<int>(t);
  o.kb0 = static_cast<int>(lo - t * p.kblocks);
  o.kb1 = static_cast<int>(hi - t * p.kblocks);
  const int64_t cf = ds_owner(t * p.kblocks, T, G);
  const int64_t cl = ds_owner((t + 1) * p.kblocks - 1, T, G);
  o.cfirst = static_cast<int>(cf);
  o.nslots = static_cast<int>(cl - cf + 1);
  o.seg = u;
  return true;
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <typename T>
__device__ __forceinline__ float ds_f32(T x);
template <>
__device__ __forceinline__ float ds_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float ds_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T ds_t16(float x);
template <>
__device__ __forceinline__ __half ds_t16<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 ds_t16<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Activation block of the prep buffer and of a stage (bytes): the fragments
// [4 chunks][M rows][4 quad columns][16 B], then the row sums [8*NJ] x 4 B.
__host__ __device__ __forceinline__ uint32_t ds_ablk(int nj, int m) {
  return static_cast<uint32_t>(m) * 256 + 32 * nj;
}

// Stage layout (bytes, every part 16-byte aligned):
//   W [sb][4 chunks][128 rows][16]   prepacked nibbles of the stage's K blocks
//   A [sb][ds_ablk]                  activation fragments + block row sums
//   C [sb][256]                      scale row (128 x 16-bit, or 128 x int8)
//   Z [sb][256]                      zero-point row
struct DsLayout {
  uint32_t w, a, c, z, stage;
};
__host__ __device__ __forceinline__ DsLayout ds_layout(int sb, int nj, int m) {
  DsLayout l;
  l.w = 0;
  l.a = l.w + sb * kWBlk;
  l.c = l.a + sb * ds_ablk(nj, m);
  l.z = l.c + sb * 256;
  l.stage = l.z + sb * 256;
  return l;
}

}  // namespace

size_t ds_smem_bytes(int sb, int nj, int m, int stages) {
  return static_cast<size_t>(ds_layout(sb, nj, m).stage) * stages + 2 * 8 * stages + 16;
}
size_t ds_prep_bytes(int nj, int m, int kblocks) {
  return static_cast<size_t>(ds_ablk(nj, m)) * kblocks;
}

// ---------------------------------------------------------------- ds_prep
// One CTA per 128-K block, 128*NJ threads: thread (c, j, lane) writes the
// 16-byte fragment of activation row m = j*8 + lane/4 (m < M), K = 32c +
// 8*(lane%4) + 0..7 (zeros past K), and its part of the block row sums,
// reduced in a fixed order.
template <int MODE, int NJ>
__global__ void __launch_bounds__(128 * NJ) ds_prep_kernel(const void* __restrict__ act,
                                                            int64_t M, int64_t K,
                                                            uint8_t* __restrict__ prep) {
  // let the dependent GEMM launch now: its weight stream does not need us
  asm volatile("griddepcontrol.launch_dependents;");
  // the previous kernel of the stream (which may produce the activations, and
  // the previous call's GEMM, which reads this buffer) is complete
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr bool F16 = MODE == kW4A16_F16;
  using T16 = typename std::conditional<F16, __half, __nv_bfloat16>::type;
  __shared__ float fpart[4][NJ][32];
  __shared__ int ipart[4][NJ][32];
  const int kb = blockIdx.x;
  const int lane = threadIdx.x & 31, j = (threadIdx.x >> 5) % NJ, c = threadIdx.x / (32 * NJ);
  const int64_t m = j * 8 + (lane >> 2);
  const int64_t k0 = static_cast<int64_t>(kb) * kBlkK + 32 * c + 8 * (lane & 3);
  uint8_t* blk = prep + static_cast<int64_t>(kb) * ds_ablk(NJ, static_cast<int>(M));
  uint4 v = make_uint4(0, 0, 0, 0);
  float fs = 0.f;
  int is = 0;
  if (m < M && k0 < K) {  // K % 64 == 0: the 8 values are all inside or all outside
    // fp16 fragments (W4A8, f16): the values of odd pairs (positions 2, 3, 6,
    // 7) are divided by 16, to match weights read 16x too large.  Exact for
    // int8 values; for fp16 activations exact when |a| >= 2^-10, while a
    // smaller |a| gives a subnormal quotient rounded to the nearest multiple
    // of 2^-24 (an absolute error of at most 2^-25 in that activation).
    if (MODE == kW4A8) {
      const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const int8_t*>(act) + m * K + k0);
      const int8_t* b8 = reinterpret_cast<const int8_t*>(&raw);
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float f = (h & 1) ? 0.0625f : 1.f;
        const __half2 p = __floats2half2_rn(static_cast<float>(b8[2 * h]) * f,
                                            static_cast<float>(b8[2 * h + 1]) * f);
        w[h] = *reinterpret_cast<const uint32_t*>(&p);
        is += static_cast<int>(b8[2 * h]) + static_cast<int>(b8[2 * h + 1]);
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      v = *reinterpret_cast<const uint4*>(static_cast<const T16*>(act) + m * K + k0);
      const T16* e = reinterpret_cast<const T16*>(&v);
      fs = ((ds_f32(e[0]) + ds_f32(e[1])) + (ds_f32(e[2]) + ds_f32(e[3]))) +
           ((ds_f32(e[4]) + ds_f32(e[5])) + (ds_f32(e[6]) + ds_f32(e[7])));
      if (F16) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const __half2 q16 = __float2half2_rn(0.0625f);
#pragma unroll
        for (int h = 1; h < 4; h += 2) {
          __half2 x = __hmul2(*reinterpret_cast<const __half2*>(&w[h]), q16);
          w[h] = *reinterpret_cast<const uint32_t*>(&x);
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (m < M) reinterpret_cast<uint4*>(blk)[(c * M + m) * 4 + (lane & 3)] = v;
  fpart[c][j][lane] = fs;
  ipart[c][j][lane] = is;
  __syncthreads();
  if (threadIdx.x < 8 * NJ) {
    const int jj = threadIdx.x >> 3, g = threadIdx.x & 7;
    uint32_t* sums = reinterpret_cast<uint32_t*>(blk + M * 256);
    if (MODE == kW4A8) {
      int s = 0;
      for (int cc = 0; cc < 4; ++cc)
        for (int t = 0; t < 4; ++t) s += ipart[cc][jj][g * 4 + t];
      sums[threadIdx.x] = static_cast<uint32_t>(s);
    } else {
      float s = 0.f;
      for (int cc = 0; cc < 4; ++cc)
        s += (fpart[cc][jj][g * 4] + fpart[cc][jj][g * 4 + 1]) +
             (fpart[cc][jj][g * 4 + 2] + fpart[cc][jj][g * 4 + 3]);
      sums[threadIdx.x] = __float_as_uint(s);
    }
  }
}

// ---------------------------------------------------------------- ds_gemm
template <int MODE, int NJ>
__global__ void __launch_bounds__(DsShape<NJ>::Threads, ds_ctas_per_sm(NJ))
    ds_gemm_kernel(const DsPlan p, const TcArgs args, const uint8_t* __restrict__ prep) {
  constexpr int kDsRP = DsShape<NJ>::RP, kDsCols = DsShape<NJ>::Cols;
  constexpr int kDsConsumers = DsShape<NJ>::Consumers;
  constexpr int kDsWProd = DsShape<NJ>::WProd, kDsAProd = DsShape<NJ>::AProd;
  constexpr bool F16 = MODE == kW4A16_F16;
  using T16 = typename std::conditional<F16, __half, __nv_bfloat16>::type;
  extern __shared__ __align__(128) uint8_t smem[];
  const int SB = kDsSB, S = p.stages;
  const int64_t M = args.M, N = args.N, K = args.K;
  const DsLayout L = ds_layout(SB, NJ, static_cast<int>(M));
  const uint32_t ablk = ds_ablk(NJ, static_cast<int>(M));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(L.stage) * S);
  uint64_t* empty = full + S;
  volatile int* abort = reinterpret_cast<int*>(empty + S);
  const uint32_t sbase = smem_addr(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 2);  // weight producer + activation producer
      mbar_init(&empty[i], kDsConsumers);
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int64_t chunks = K / kChunkK;
  const bool pc = args.group_size >= K;  // one scale group per column
  const int esz = MODE == kW4A8 ? 1 : 2;

  if (warp == kDsWProd || warp == kDsAProd) {
    // --------------------------------------------------------- producers
    if (lane == 0) {
      const bool wprod = warp == kDsWProd;
      if (!wprod) asm volatile("griddepcontrol.wait;" ::: "memory");  // ds_prep is complete
      uint32_t it = 0, s = 0, ph = 0;  // stage count, it % S, (it / S) & 1
      bool ok = true;
      DsUnit u;
      // K blocks per scale group (one division per unit below, none per block)
      const int bpg = pc ? 1 : static_cast<int>(args.group_size / kBlkK);
      for (int ui = 0; ok && ds_unit(p, ui, u); ++ui) {
        const int64_t n0 = static_cast<int64_t>(u.tile) * kTileN;
        const uint32_t ncol = static_cast<uint32_t>(N - n0 < kTileN ? N - n0 : kTileN);
        const uint32_t scb = (!pc && args.scales) ? ncol * esz : 0;
        const uint32_t zpb = (!pc && args.zeros) ? ncol * esz : 0;
        const uint8_t* wtile = args.b_packed + static_cast<int64_t>(u.tile) * chunks * (kTileN * 16);
        int64_t gcur = u.kb0 / bpg;          // scale group of the next block
        int gleft = bpg - u.kb0 % bpg;       // blocks left in it
        for (int kb = u.kb0; kb < u.kb1; kb += SB, ++it) {
          if (!mbar_wait(&empty[s], ph ^ 1, abort, args.status)) {
            ok = false;
            break;
          }
          const int nb = u.kb1 - kb < SB ? u.kb1 - kb : SB;
          const uint32_t st = sbase + s * L.stage, bar = smem_addr(&full[s]);
          if (wprod) {
            int64_t nch = chunks - static_cast<int64_t>(kb) * 4;
            if (nch > 4 * nb) nch = 4 * nb;
            const uint32_t wb = static_cast<uint32_t>(nch) * (kTileN * 16);
            mbar_arrive_expect_tx(&full[s], wb + nb * (scb + zpb));
            bulk_g2s_a(st + L.w, wtile + static_cast<int64_t>(kb) * kWBlk, wb, bar);
            for (int b = 0; b < nb && (scb || zpb); ++b) {
              const int64_t g = gcur;
              if (--gleft == 0) {
                ++gcur;
                gleft = bpg;
              }
              if (scb)
                bulk_g2s_a(st + L.c + b * 256,
                           static_cast<const uint8_t*>(args.scales) + (g * N + n0) * esz, scb, bar);
              if (zpb)
                bulk_g2s_a(st + L.z + b * 256,
                           static_cast<const uint8_t*>(args.zeros) + (g * N + n0) * esz, zpb, bar);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], nb * ablk);
            bulk_g2s_a(st + L.a, prep + static_cast<int64_t>(kb) * ablk, nb * ablk, bar);
          }
          if (++s == static_cast<uint32_t>(S)) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // every copy issued lands before the CTA may exit
      for (uint32_t j = (it > static_cast<uint32_t>(S) ? it - S : 0); j < it; ++j) {
        volatile int no_abort = 0;
        mbar_wait(&full[j % S], (j / S) & 1, &no_abort, args.status);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  asm volatile("griddepcontrol.launch_dependents;");  // ds_reduce may launch and wait
  const int w = warp, g = lane >> 2, t = lane & 3;
  // fp16 MMA (W4A8, f16): a word's nibble pairs sit at bits 0-3 / 4-7 (and,
  // after one shift, 8-11 / 12-15) of each half; OR-ed into the mantissa of
  // 1024 they read as 1024 + q and 1024 + 16q, exact.  Subtracting
  // 1024 + bias and 1024 + 16*bias leaves q - bias and 16*(q - bias); the
  // activations of the second kind of pair were divided by 16 when staged.
  // bf16 MMA (W4A16 bf16): the 7-bit mantissa holds one nibble, at bits 0-3
  // (128 + q); the offset 128 + bias is folded out with the block row sums.
  constexpr bool kFp16Mma = MODE != kW4A16_BF16;
  const uint32_t magic = kFp16Mma ? 0x64006400u : 0x43004300u;
  const float mb = 128.f + static_cast<float>(args.wbias);  // bf16 fold offset
  uint32_t off_lo = 0, off_hi = 0;
  if (kFp16Mma) {
    const __half2 lo = __float2half2_rn(1024.f + static_cast<float>(args.wbias));
    const __half2 hi = __float2half2_rn(1024.f + 16.f * static_cast<float>(args.wbias));
    off_lo = *reinterpret_cast<const uint32_t*>(&lo);
    off_hi = *reinterpret_cast<const uint32_t*>(&hi);
  }
  // ldmatrix row address of this lane: matrix (chunk) lane/8, row lane%8
  const uint32_t ldsm_off = (lane >> 3) * 2048 + (kDsCols * w + (lane & 7)) * 16;
  bool live[NJ];
  uint32_t aoff[NJ];  // activation fragment of row j*8 + g, quad column t
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    live[j] = j * 8 + g < M;
    aoff[j] = static_cast<uint32_t>((j * 8 + g) * 64 + t * 16);
  }
  const uint32_t a_chunk = static_cast<uint32_t>(M) * 64;  // fragment bytes per chunk
  constexpr int MR = 8 * NJ;                               // rows of a partial slot
  const size_t slot_elems = static_cast<size_t>(MR) * kTileN;
  // K blocks folded together: one scale group; with one group per column a
  // run whose fp32 sums stay exact integers below 2^24 (W4A8: 64 blocks of
  // 128 products |a * (q - bias)| <= 128 * 8), or the whole tile segment
  // (W4A16).
  const int fold_blocks =
      pc ? (MODE == kW4A8 ? 64 : (1 << 30)) : static_cast<int>(args.group_size / kBlkK);
  auto store = [&](int64_t m, int64_t n, float vf, int32_t vi) {
    if (m >= M || n >= N) return;
    store_out<MODE>(args, m, n, vf, vi);
  };

  uint32_t it = 0, cs = 0, cph = 0;  // stage count, it % S, (it / S) & 1
  bool ok = true;
  DsUnit u;
  for (int ui = 0; ok && ds_unit(p, ui, u); ++ui) {
    const int64_t n0 = static_cast<int64_t>(u.tile) * kTileN;
    float res[kDsRP][NJ][4];
    int32_t ires[kDsRP][NJ][4];
    float acc[2][kDsRP][NJ][4];  // [MMA parity h][R][j][e]: independent chains
    float fsum[NJ][2];           // row sums of the blocks since the last fold
    int isum[NJ][2];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        fsum[j][e] = 0.f;
        isum[j][e] = 0;
      }
#pragma unroll
      for (int R = 0; R < kDsRP; ++R)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          res[R][j][e] = 0.f;
          ires[R][j][e] = 0;
          acc[0][R][j][e] = 0.f;
          acc[1][R][j][e] = 0.f;
        }
    }
    // scale / zero-point of row groups q (columns n0 + kDsCols*w + 8q + g)
    float sq[2 * kDsRP], cq[2 * kDsRP];
    int isq[2 * kDsRP];
    if (pc) {
#pragma unroll
      for (int q = 0; q < 2 * kDsRP; ++q) {
        const int64_t n = n0 + kDsCols * w + 8 * q + g;
        const bool in = n < N;
        if (MODE == kW4A8) {
          isq[q] = 1;
          sq[q] = 1.f;
          cq[q] = 0.f;
        } else {
          sq[q] = in ? ds_f32(static_cast<const T16*>(args.scales)[n]) : 0.f;
          const float z = (in && args.zeros) ? ds_f32(static_cast<const T16*>(args.zeros)[n]) : 0.f;
          cq[q] = kFp16Mma ? z : fmaf(mb, sq[q], z);
        }
      }
    }
    // blocks to go before the next fold (scale groups are aligned to K = 0)
    int fleft = pc ? fold_blocks : fold_blocks - u.kb0 % fold_blocks;
    for (int kb = u.kb0; kb < u.kb1; kb += kDsSB, ++it) {
      const uint32_t s = cs;
      if (!mbar_wait(&full[s], cph, abort, args.status)) {
        ok = false;
        break;
      }
      if (++cs == static_cast<uint32_t>(S)) {
        cs = 0;
        cph ^= 1;
      }
      const uint32_t st = sbase + s * L.stage;
      const uint8_t* stp = smem + static_cast<size_t>(s) * L.stage;
#pragma unroll
      for (int b = 0; b < kDsSB; ++b) {
        const int kbb = kb + b;
        if (kbb >= u.kb1) break;
        uint32_t x[2 * kDsRP][4];  // [row group q][chunk c]: word t of row kDsCols*w + 8q + g
#pragma unroll
        for (int q = 0; q < 2 * kDsRP; ++q)
          ldsm_x4(st + L.w + b * kWBlk + ldsm_off + q * 128, x[q]);
        const uint32_t ab = st + L.a + b * ablk;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 v[NJ];  // this chunk's activation fragments
#pragma unroll
          for (int j = 0; j < NJ; ++j)
            v[j] = live[j] ? lds128(ab + c * a_chunk + aoff[j]) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int R = 0; R < kDsRP; ++R) {
              const uint32_t xa = x[2 * R][c] >> (8 * h), xb = x[2 * R + 1][c] >> (8 * h);
              uint32_t a0, a1, a2, a3;
              if constexpr (kFp16Mma) {
                const __half2 lo = *reinterpret_cast<const __half2*>(&off_lo);
                const __half2 hi = *reinterpret_cast<const __half2*>(&off_hi);
                uint32_t p0 = lop_and_or(xa, 0x000F000Fu, magic);
                uint32_t p1 = lop_and_or(xb, 0x000F000Fu, magic);
                uint32_t p2 = lop_and_or(xa, 0x00F000F0u, magic);
                uint32_t p3 = lop_and_or(xb, 0x00F000F0u, magic);
                __half2 r0 = __hsub2(*reinterpret_cast<__half2*>(&p0), lo);
                __half2 r1 = __hsub2(*reinterpret_cast<__half2*>(&p1), lo);
                __half2 r2 = __hsub2(*reinterpret_cast<__half2*>(&p2), hi);
                __half2 r3 = __hsub2(*reinterpret_cast<__half2*>(&p3), hi);
                a0 = *reinterpret_cast<uint32_t*>(&r0);
                a1 = *reinterpret_cast<uint32_t*>(&r1);
                a2 = *reinterpret_cast<uint32_t*>(&r2);
                a3 = *reinterpret_cast<uint32_t*>(&r3);
              } else {
                a0 = lop_and_or(xa, 0x000F000Fu, magic);
                a1 = lop_and_or(xb, 0x000F000Fu, magic);
                a2 = lop_and_or(xa >> 4, 0x000F000Fu, magic);
                a3 = lop_and_or(xb >> 4, 0x000F000Fu, magic);
              }
#pragma unroll
              for (int j = 0; j < NJ; ++j) {
                const uint32_t b0 = h ? v[j].z : v[j].x;
                const uint32_t b1 = h ? v[j].w : v[j].y;
                mma16816<kFp16Mma>(acc[h][R][j], a0, a1, a2, a3, b0, b1);
              }
            }
        }
        // block row sums
        const uint8_t* sums = stp + L.a + b * ablk + M * 256;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const uint2 S2 = *reinterpret_cast<const uint2*>(sums + (j * 8 + 2 * t) * 4);
          if (MODE == kW4A8) {
            isum[j][0] += static_cast<int>(S2.x);
            isum[j][1] += static_cast<int>(S2.y);
          } else {
            fsum[j][0] += __uint_as_float(S2.x);
            fsum[j][1] += __uint_as_float(S2.y);
          }
        }
        if (!pc) {  // the group's scale (and zero-point) rows
#pragma unroll
          for (int q = 0; q < 2 * kDsRP; ++q) {
            const int row = kDsCols * w + 8 * q + g;
            if (MODE == kW4A8) {
              isq[q] = args.scales
                           ? static_cast<int>(reinterpret_cast<const int8_t*>(stp + L.c + b * 256)[row])
                           : 1;
            } else {
              sq[q] = ds_f32(reinterpret_cast<const T16*>(stp + L.c + b * 256)[row]);
              const float z = args.zeros
                                  ? ds_f32(reinterpret_cast<const T16*>(stp + L.z + b * 256)[row])
                                  : 0.f;
              cq[q] = kFp16Mma ? z : fmaf(mb, sq[q], z);
            }
          }
        }
        // fold at the end of a scale group / exact run, and of the segment
        if (--fleft == 0) fleft = fold_blocks;
        if (kbb + 1 == u.kb1 || fleft == fold_blocks) {
#pragma unroll
          for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int R = 0; R < kDsRP; ++R)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int q = 2 * R + (e >> 1);
                const float a = acc[0][R][j][e] + acc[1][R][j][e];
                acc[0][R][j][e] = 0.f;
                acc[1][R][j][e] = 0.f;
                if (MODE == kW4A8) {
                  const int blk = __float2int_rn(a);  // exact: sum of a * (q - bias)
                  ires[R][j][e] += pc ? blk : isq[q] * blk;
                } else {
                  res[R][j][e] = fmaf(sq[q], a, fmaf(-cq[q], fsum[j][e & 1], res[R][j][e]));
                }
              }
#pragma unroll
          for (int j = 0; j < NJ; ++j) {
            fsum[j][0] = fsum[j][1] = 0.f;
            isum[j][0] = isum[j][1] = 0;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok) break;

    // ---- this tile's result: the output, or a partial slot for ds_reduce
    if (u.nslots == 1) {
#pragma unroll
      for (int R = 0; R < kDsRP; ++R)
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            store(j * 8 + 2 * t + (e & 1), n0 + kDsCols * w + 16 * R + g + 8 * (e >> 1),
                  res[R][j][e], ires[R][j][e]);
      continue;
    }
    const size_t mine = (static_cast<size_t>(blockIdx.x) * p.max_segs + u.seg) * slot_elems;
#pragma unroll
    for (int R = 0; R < kDsRP; ++R)
#pragma unroll
      for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const size_t off = mine + static_cast<size_t>(j * 8 + 2 * t + (e & 1)) * kTileN +
                             kDsCols * w + 16 * R + g + 8 * (e >> 1);
          if (MODE == kW4A8) static_cast<int32_t*>(args.partials)[off] = ires[R][j][e];
          else static_cast<float*>(args.partials)[off] = res[R][j][e];
        }
  }
}

// -------------------------------------------------------------- ds_reduce
// Tiles that several CTAs share get the sum of their partial slots, added in
// K order (deterministic): one thread per output element, a CTA covers two
// rows of one 128-column tile.  Launched as a programmatic dependent of
// ds_gemm; waits for it to complete.
constexpr int kDsRedRows = 2;
constexpr int kDsRedThreads = kDsRedRows * kTileN;
constexpr int kDsRedMaxSlots = 64;  // slot offsets kept in shared memory

template <int MODE, int NJ>
__global__ void __launch_bounds__(kDsRedThreads) ds_reduce_kernel(const DsPlan p, const TcArgs args) {
  asm volatile("griddepcontrol.launch_dependents;");  // the next call may start its prologue
  asm volatile("griddepcontrol.wait;" ::: "memory");  // ds_gemm is complete
  using T16 = typename std::conditional<MODE == kW4A16_F16, __half, __nv_bfloat16>::type;
  __shared__ unsigned long long sbase[kDsRedMaxSlots];
  const int64_t T = static_cast<int64_t>(p.n_tiles) * p.kblocks, G = p.grid;
  const int tile = blockIdx.x;
  const int64_t cf = ds_owner(static_cast<int64_t>(tile) * p.kblocks, T, G);
  const int64_t cl = ds_owner((static_cast<int64_t>(tile) + 1) * p.kblocks - 1, T, G);
  const int nslots = static_cast<int>(cl - cf + 1);
  if (nslots == 1) return;
  const size_t slot_elems = static_cast<size_t>(8 * NJ) * kTileN;
  auto slot_base = [&](int sl) -> unsigned long long {
    const int64_t cpr = cf + sl;
    const int64_t seg = tile - div_nn(ds_start(cpr, T, G), p.kblocks);
    return (static_cast<size_t>(cpr) * p.max_segs + seg) * slot_elems;
  };
  for (int sl = threadIdx.x; sl < nslots && sl < kDsRedMaxSlots; sl += kDsRedThreads)
    sbase[sl] = slot_base(sl);
  __syncthreads();
  const int64_t M = args.M, N = args.N;
  const int m = blockIdx.y * kDsRedRows + threadIdx.x / kTileN, col = threadIdx.x % kTileN;
  const int64_t n = static_cast<int64_t>(tile) * kTileN + col;
  if (m >= M || n >= N) return;
  const uint32_t* part = static_cast<const uint32_t*>(args.partials);
  const size_t off = static_cast<size_t>(m) * kTileN + col;
  float af = 0.f;
  int32_t ai = 0;
  constexpr int kBatch = 8;  // slot loads in flight together
  for (int s0 = 0; s0 < nslots; s0 += kBatch) {
    uint32_t x[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int sl = s0 + q;
      x[q] = sl < nslots ? part[(sl < kDsRedMaxSlots ? sbase[sl] : slot_base(sl)) + off] : 0u;
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int sl = s0 + q;
      if (sl >= nslots) break;
      if (MODE == kW4A8) ai += static_cast<int32_t>(x[q]);
      else af = sl == 0 ? __uint_as_float(x[q]) : af + __uint_as_float(x[q]);
    }
  }
  store_out<MODE>(args, m, n, af, ai);
}

namespace {
template <int MODE, int NJ>
cudaError_t launch_ds_t(const DsPlan& plan, const void* a, const TcArgs& args, uint8_t* prep,
                        cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3(plan.kblocks);
  pcfg.blockDim = dim3(128 * NJ);
  pcfg.stream = s;
  pcfg.attrs = attr;
  pcfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&pcfg, &ds_prep_kernel<MODE, NJ>, a, args.M, args.K, prep);
  if (e != cudaSuccess) return e;
  auto fn = &ds_gemm_kernel<MODE, NJ>;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(plan.smem_bytes));
  if (e != cudaSuccess) return e;
  static const bool debug = getenv("W4_DEBUG") != nullptr;
  if (debug) {
    int blocks = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, DsShape<NJ>::Threads,
                                                  plan.smem_bytes);
    fprintf(stderr, "w4: ds resident CTAs per SM: %d (smem %zu)\n", blocks, plan.smem_bytes);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(DsShape<NJ>::Threads);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fn, plan, args, static_cast<const uint8_t*>(prep));
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(plan.n_tiles, static_cast<unsigned>((args.M + kDsRedRows - 1) / kDsRedRows));
  cfg.blockDim = dim3(kDsRedThreads);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, &ds_reduce_kernel<MODE, NJ>, plan, args);
}
}  // namespace

cudaError_t launch_ds(const DsPlan& plan, const void* a, const TcArgs& args, uint8_t* prep,
                      cudaStream_t s) {
  if (plan.nj == 1) {
    if (plan.mode == kW4A16_F16) return launch_ds_t<kW4A16_F16, 1>(plan, a, args, prep, s);
    if (plan.mode == kW4A16_BF16) return launch_ds_t<kW4A16_BF16, 1>(plan, a, args, prep, s);
    return launch_ds_t<kW4A8, 1>(plan, a, args, prep, s);
  }
  if (plan.nj == 2) {
    if (plan.mode == kW4A16_F16) return launch_ds_t<kW4A16_F16, 2>(plan, a, args, prep, s);
    if (plan.mode == kW4A16_BF16) return launch_ds_t<kW4A16_BF16, 2>(plan, a, args, prep, s);
    return launch_ds_t<kW4A8, 2>(plan, a, args, prep, s);
  }
  if (plan.mode == kW4A16_F16) return launch_ds_t<kW4A16_F16, 4>(plan, a, args, prep, s);
  if (plan.mode == kW4A16_BF16) return launch_ds_t<kW4A16_BF16, 4>(plan, a, args, prep, s);
  return launch_ds_t<kW4A8, 4>(plan, a, args, prep, s);
}

}  // namespace w4
