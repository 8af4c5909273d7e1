// w4_gv.cu — the clustered skinny-M ("decode") schedule of the 4-bit-weight
// GEMM: up to 32 activation rows, HBM-bound on the weight bytes, in ONE
// launch with no global scratch.
//
// Decomposition: every 128-column weight tile is split along K over a
// thread-block cluster of C CTAs (C = 1..16, chosen on the host so that all
// n_tiles x C CTAs are resident at once and every CTA streams the same number
// of 128-K blocks).  Each CTA streams its contiguous K range of the tile
// through a ring of shared-memory stages:
//   producer thread : one bulk copy of the block's prepacked nibbles (8 KB),
//                     the block's scale / zero-point rows (per-group
//                     weights), and one TMA box of the block's activations
//                     (all rows of the problem, 128-byte swizzled); the
//                     weight copies of the first stages leave before the CTA
//                     does anything else, and only the activation copies
//                     wait for the grid this one may overlap (programmatic
//                     dependent launch).
//   consumer warps  : ldmatrix hands every thread word t of its weight rows'
//                     32-K chunks; each nibble pair becomes a 16-bit pair
//                     (magic + q) with one shift and one lop3 (exact), and
//                     warp-level mma.sync.m16n8k16 accumulates a K block in
//                     fp32.  The block is folded into the running result with
//                     its scale and zero-point:
//
//                       sum_k a*w_hat = s*(sum_k a*(magic+q) - (magic+bias)*S) - w_z*S
//
//                     (S: the block's activation row sums, which the
//                     consumers add up from the fragments they load), the
//                     per-element rule w_hat = (q - bias)*s - w_z of the
//                     Machete Readme ("Overview") applied once per block.
//                     W4A8 (pytorch/ao PR #1113 "support W4A8 Marlin kernel")
//                     and fp16 activations use fp16 MMAs with two nibble
//                     fields per half (1024 + q and 1024 + 16q, the second
//                     kind of pair met by activations divided by 16) and
//                     subtract the offset exactly before the MMA; W4A8 block
//                     sums are exact integers.
// Split-K reduction: every CTA of a cluster writes its 128 x rows partial
// sums to its own shared memory; after a cluster barrier, CTA r adds the
// partial sums of its slice of the tile's columns from all C CTAs through
// distributed shared memory, in rank order (= K order: deterministic), and
// writes the outputs; a second cluster barrier keeps every CTA's shared
// memory alive until the others have read it.
//
// K order inside a 128-K block: thread t of an MMA quad holds word t of each
// 32-K chunk c, i.e. K = 32c + 8t + 0..7, which is also 16 contiguous bytes
// of a row-major activation row: the activation fragments are read straight
// from the TMA tile.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdio>
#include <cstdlib>

#include "w4_epilogue.cuh"
#include "w4_internal.h"
#include "w4_ptx.cuh"

namespace w4 {
namespace {

// A consumer warp owns RP pairs of 8-row weight groups (16 weight columns per
// pair, one m16n8k16 A tile): 32 columns for up to 16 activation rows (four
// consumer warps), 16 for up to 32 rows (eight warps, so that the
// accumulators of four 8-row activation tiles fit in registers).
template <int NJ>
struct GvShape {
  static constexpr int RP = NJ >= 4 ? 1 : 2;
  static constexpr int Cols = 16 * RP;
  static constexpr int Consumers = kTileN / Cols;
  static constexpr int Prod = Consumers;  // producer warp
  static constexpr int Threads = 32 * (Consumers + 1);
};
constexpr int kGvBlkK = 128;
constexpr uint32_t kGvWBlk = 4 * kTileN * 16;  // prepacked bytes of one K block of a tile

__device__ __forceinline__ uint32_t gv_lop(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ void gv_ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint4 gv_lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 gv_lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
template <bool F16>
__device__ __forceinline__ void gv_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
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

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_dsmem(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <typename T>
__device__ __forceinline__ float gv_f32(T x);
template <>
__device__ __forceinline__ float gv_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float gv_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T gv_t16(float x);
template <>
__device__ __forceinline__ __half gv_t16<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 gv_t16<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Eight int8 activations (two words) as four fp16 pairs, the second and
// fourth pair divided by 16: each byte is moved into the low byte of a
// 16-bit lane (prmt), its sign bit flipped and 0x64 placed above it (one
// lop3), which reads as 1024 + 128 + x in fp16; subtracting 1152, or
// multiplying by 1/16 and subtracting 72, is exact.
__device__ __forceinline__ uint4 gv_i8x8_to_f16(uint2 raw) {
  uint32_t p[4];
  asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(p[0]) : "r"(raw.x));
  asm("prmt.b32 %0, %1, 0, 0x4342;" : "=r"(p[1]) : "r"(raw.x));
  asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(p[2]) : "r"(raw.y));
  asm("prmt.b32 %0, %1, 0, 0x4342;" : "=r"(p[3]) : "r"(raw.y));
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t r;
    // (p ^ 0x00800080) | 0x64006400
    asm("lop3.b32 %0, %1, %2, %3, 0x1E;" : "=r"(r) : "r"(p[i]), "r"(0x00800080u), "r"(0x64006400u));
    h[i] = r;
  }
  const __half2 k1152 = __float2half2_rn(1152.f), k16 = __float2half2_rn(0.0625f),
                k72 = __float2half2_rn(-72.f);
  __half2 r0 = __hsub2(*reinterpret_cast<__half2*>(&h[0]), k1152);
  __half2 r1 = __hfma2(*reinterpret_cast<__half2*>(&h[1]), k16, k72);
  __half2 r2 = __hsub2(*reinterpret_cast<__half2*>(&h[2]), k1152);
  __half2 r3 = __hfma2(*reinterpret_cast<__half2*>(&h[3]), k16, k72);
  return make_uint4(*reinterpret_cast<uint32_t*>(&r0), *reinterpret_cast<uint32_t*>(&r1),
                    *reinterpret_cast<uint32_t*>(&r2), *reinterpret_cast<uint32_t*>(&r3));
}

// Eight E4M3 activations (two words) as four fp16 pairs (exact: every E4M3
// value is an fp16 value), the second and fourth pair divided by 16 (exact:
// the quotients are multiples of 2^-13 of magnitude at most 28).
__device__ __forceinline__ uint4 gv_e4m3x8_to_f16(uint2 raw) {
  uint32_t h[4];
  const uint16_t b[4] = {static_cast<uint16_t>(raw.x), static_cast<uint16_t>(raw.x >> 16),
                         static_cast<uint16_t>(raw.y), static_cast<uint16_t>(raw.y >> 16)};
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[i]) : "h"(b[i]));
  const __half2 k16 = __float2half2_rn(0.0625f);
  __half2 r1 = __hmul2(*reinterpret_cast<__half2*>(&h[1]), k16);
  __half2 r3 = __hmul2(*reinterpret_cast<__half2*>(&h[3]), k16);
  return make_uint4(h[0], *reinterpret_cast<uint32_t*>(&r1), h[2], *reinterpret_cast<uint32_t*>(&r3));
}

}  // namespace

// Shared-memory layout: S stages of [W 8 KB][A rows x 128 K], then S scale /
// zero-point row pairs [C 256 B][Z 256 B], the partial-sum tile of the
// cluster reduction [8*NJ][128] x 4 B, and the barriers.  Every A tile
// starts on a 1024-byte boundary (128-byte swizzle).
__host__ __device__ inline uint32_t gv_act_bytes(int nj, int mode) {
  return (mode == kW4A8 || mode == kW4A8F8 ? 128u : 256u) * 8u * static_cast<uint32_t>(nj);
}
__host__ __device__ inline uint32_t gv_stage_bytes(int nj, int mode) {
  return kGvWBlk + gv_act_bytes(nj, mode);
}
size_t gv_smem_bytes(int nj, int mode, int stages) {
  return 1024 + static_cast<size_t>(stages) * (gv_stage_bytes(nj, mode) + 512) +
         static_cast<size_t>(8 * nj) * kTileN * 4 + 2 * 8 * stages + 16;
}

template <int MODE, int NJ>
__global__ void __launch_bounds__(GvShape<NJ>::Threads, gv_ctas_per_sm(NJ))
    gv_gemm_kernel(const __grid_constant__ CUtensorMap amap, const GvPlan p, const TcArgs args) {
  constexpr int RP = GvShape<NJ>::RP, Cols = GvShape<NJ>::Cols;
  constexpr int Consumers = GvShape<NJ>::Consumers, Prod = GvShape<NJ>::Prod;
  constexpr bool F16 = MODE == kW4A16_F16;
  using T16 = typename std::conditional<F16, __half, __nv_bfloat16>::type;
  // fp16 MMAs with the offset subtracted before the MMA (W4A8, fp16
  // activations); bf16 MMAs with the offset folded out with the row sums
  constexpr bool kFp16Mma = MODE != kW4A16_BF16;
  constexpr bool k8Bit = MODE == kW4A8 || MODE == kW4A8F8;  // 1-byte activations
  constexpr uint32_t kActBytes = (k8Bit ? 128u : 256u) * 8u * NJ;
  constexpr uint32_t kStage = kGvWBlk + kActBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  uint8_t* cz = smem + static_cast<size_t>(S) * kStage;          // [S][512]
  uint32_t* red = reinterpret_cast<uint32_t*>(cz + static_cast<size_t>(S) * 512);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 8 * NJ * kTileN);
  uint64_t* empty = full + S;
  volatile int* abort = reinterpret_cast<int*>(empty + S);
  const uint32_t sbase = smem_addr(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t M = args.M, N = args.N, K = args.K;
  const int C = p.cluster;
  const int tile = blockIdx.x / C, rank = blockIdx.x - tile * C;
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.kblocks / C);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.kblocks / C);
  const int nkb = kb1 - kb0;
  const int64_t n0 = static_cast<int64_t>(tile) * kTileN;
  const int64_t chunks = K / kChunkK;
  const bool pc = args.group_size >= K;  // one scale group per column
  const int esz = MODE == kW4A8 ? 1 : 2;
  const uint32_t ncol = static_cast<uint32_t>(N - n0 < kTileN ? N - n0 : kTileN);
  const uint32_t scb = (!pc && args.scales) ? ncol * esz : 0;
  const uint32_t zpb = (!pc && args.zeros) ? ncol * esz : 0;
  const int bpg = pc ? 1 : static_cast<int>(args.group_size / kGvBlkK);  // K blocks per group
  const uint8_t* wtile = args.b_packed + static_cast<int64_t>(tile) * chunks * (kTileN * 16);
  auto wbytes = [&](int kb) -> uint32_t {
    int64_t nch = chunks - static_cast<int64_t>(kb) * 4;
    if (nch > 4) nch = 4;
    return static_cast<uint32_t>(nch) * (kTileN * 16);
  };
  // weights (and scale / zero rows) of K block kb into stage s
  auto issue_w = [&](int kb, int s) {
    const uint32_t bar = smem_addr(&full[s]);
    const uint32_t wb = wbytes(kb);
    mbar_arrive_expect_tx_a(bar, wb + scb + zpb + kActBytes);
    bulk_g2s_a(sbase + s * kStage, wtile + static_cast<int64_t>(kb) * kGvWBlk, wb, bar);
    if (scb || zpb) {
      const int64_t g = kb / bpg;
      const uint32_t czs = smem_addr(cz + s * 512);
      if (scb)
        bulk_g2s_a(czs, static_cast<const uint8_t*>(args.scales) + (g * N + n0) * esz, scb, bar);
      if (zpb)
        bulk_g2s_a(czs + 256, static_cast<const uint8_t*>(args.zeros) + (g * N + n0) * esz, zpb,
                   bar);
    }
  };
  // the activation box of K block kb into stage s (all rows; rows >= M read
  // as zeros)
  auto issue_a = [&](int kb, int s) {
    const uint32_t bar = smem_addr(&full[s]);
    const uint32_t dst = sbase + s * kStage + kGvWBlk;
    if (k8Bit) tma_load_2d_a(dst, &amap, kb * kGvBlkK, 0, bar);
    else tma_load_3d_a(dst, &amap, 0, 0, 2 * kb, bar);
  };

  if (warp == Prod && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], Consumers);
    }
    *abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&amap);
    // the first stages' weights leave before anything else happens
    const int npre = nkb < S ? nkb : S;
    for (int i = 0; i < npre; ++i) issue_w(kb0 + i, i);
  }
  __syncthreads();

  if (warp == Prod) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // activations may come from the grid this one overlaps
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const int npre = nkb < S ? nkb : S;
      for (int i = 0; i < npre; ++i) issue_a(kb0 + i, i);
      uint32_t s = npre % S, ph = npre >= S ? 1u : 0u;
      if (npre < S) s = npre;
      for (int it = npre; it < nkb; ++it) {
        if (!mbar_wait(&empty[s], ph ^ 1, abort, args.status)) break;
        issue_w(kb0 + it, s);
        issue_a(kb0 + it, s);
        if (++s == static_cast<uint32_t>(S)) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    asm volatile("griddepcontrol.launch_dependents;");
    const int w = warp, g = lane >> 2, t = lane & 3;
    const uint32_t magic = kFp16Mma ? 0x64006400u : 0x43004300u;
    const float mb = 128.f + static_cast<float>(args.wbias);  // bf16 fold offset
    uint32_t off_lo = 0, off_hi = 0;
    if (kFp16Mma) {
      const __half2 lo = __float2half2_rn(1024.f + static_cast<float>(args.wbias));
      const __half2 hi = __float2half2_rn(1024.f + 16.f * static_cast<float>(args.wbias));
      off_lo = *reinterpret_cast<const uint32_t*>(&lo);
      off_hi = *reinterpret_cast<const uint32_t*>(&hi);
    }
    // Row sums of the activations (bf16 fold, fp16 zero-points) come out of
    // one more MMA per 16-K step whose A operand is constant: ones against
    // the K values as staged, sixteens against the pairs divided by 16, so
    // that every row of D holds the activation row sums (rows 2t, 2t+1 of
    // the tile in this thread's D fragment), accumulated until the fold.
    const bool need_sum = MODE == kW4A16_BF16 || (F16 && args.zeros != nullptr);
    const uint32_t one_lo = kFp16Mma ? 0x3C003C00u : 0x3F803F80u;
    const uint32_t one_hi = kFp16Mma ? 0x4C004C00u : 0x3F803F80u;
    // ldmatrix row address of this lane: matrix (chunk) lane/8, row lane%8
    const uint32_t ldsm_off = (lane >> 3) * 2048 + (Cols * w + (lane & 7)) * 16;
    float res[RP][NJ][4];
    int32_t ires[RP][NJ][4];
    // [MMA parity h][R][j][e]: two independent chains when there are few
    // activation tiles (with four, their accumulators are independent enough)
    constexpr int H2 = NJ >= 4 ? 1 : 2;
    float acc[H2][RP][NJ][4];
    float fsum[NJ][4];        // row sums (rows j*8 + 2t, 2t+1) since the last fold
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      fsum[j][0] = fsum[j][1] = fsum[j][2] = fsum[j][3] = 0.f;
#pragma unroll
      for (int R = 0; R < RP; ++R)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          res[R][j][e] = 0.f;
          ires[R][j][e] = 0;
#pragma unroll
          for (int h = 0; h < H2; ++h) acc[h][R][j][e] = 0.f;
        }
    }
    // scale / zero-point of row groups q (columns n0 + Cols*w + 8q + g)
    float sq[2 * RP], cq[2 * RP];
    int isq[2 * RP];
#pragma unroll
    for (int q = 0; q < 2 * RP; ++q) {
      sq[q] = 1.f;
      cq[q] = 0.f;
      isq[q] = 1;
    }
    if (pc && (MODE == kW4A16_F16 || MODE == kW4A16_BF16)) {
#pragma unroll
      for (int q = 0; q < 2 * RP; ++q) {
        const int64_t n = n0 + Cols * w + 8 * q + g;
        const bool in = n < N;
        sq[q] = in ? gv_f32(static_cast<const T16*>(args.scales)[n]) : 0.f;
        const float z = (in && args.zeros) ? gv_f32(static_cast<const T16*>(args.zeros)[n]) : 0.f;
        cq[q] = kFp16Mma ? z : fmaf(mb, sq[q], z);
      }
    }
    // K blocks folded together: one scale group; with one group per column a
    // run whose fp32 sums stay exact integers below 2^24 (W4A8: 64 blocks of
    // 128 products |a * (q - bias)| <= 128 * 8), or the whole K range (W4A16)
    const int fold_blocks = pc ? (MODE == kW4A8 ? 64 : (1 << 30)) : bpg;
    int fleft = pc ? fold_blocks : fold_blocks - kb0 % fold_blocks;
    uint32_t cs = 0, cph = 0;
    bool ok = true;
    for (int it = 0; it < nkb; ++it) {
      const int kb = kb0 + it;
      const uint32_t s = cs;
      if (!mbar_wait(&full[s], cph, abort, args.status)) {
        ok = false;
        break;
      }
      if (++cs == static_cast<uint32_t>(S)) {
        cs = 0;
        cph ^= 1;
      }
      const uint32_t st = sbase + s * kStage;
      const uint32_t at = st + kGvWBlk;
      uint32_t x[2 * RP][4];  // [row group q][chunk c]: word t of row Cols*w + 8q + g
#pragma unroll
      for (int q = 0; q < 2 * RP; ++q) gv_ldsm_x4(st + ldsm_off + q * 128, x[q]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 v[NJ];  // activation fragment of row j*8 + g: K = 32c + 8t + 0..7
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int row = j * 8 + g;
          if (k8Bit) {
            // 8-bit row of 128 K: 16-byte column 2c + t/2, half t%2
            const uint2 raw = gv_lds64(at + row * 128 + ((((2 * c) | (t >> 1)) ^ g) << 4) +
                                       8 * (t & 1));
            v[j] = MODE == kW4A8 ? gv_i8x8_to_f16(raw) : gv_e4m3x8_to_f16(raw);
          } else {
            // 16-bit: half-block z = c/2 of 64 K, 16-byte column 4(c%2) + t
            const uint32_t col = static_cast<uint32_t>(((c & 1) << 2) | t);
            v[j] = gv_lds128(at + (c >> 1) * (1024u * NJ) + row * 128 + ((col ^ g) << 4));
            if constexpr (F16) {
              // the second kind of pair meets weights read 16x too large
              const __half2 q16 = __float2half2_rn(0.0625f);
              __half2 y = __hmul2(*reinterpret_cast<const __half2*>(&v[j].y), q16);
              __half2 zz = __hmul2(*reinterpret_cast<const __half2*>(&v[j].w), q16);
              v[j].y = *reinterpret_cast<uint32_t*>(&y);
              v[j].w = *reinterpret_cast<uint32_t*>(&zz);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int R = 0; R < RP; ++R) {
            const uint32_t xa = x[2 * R][c] >> (8 * h), xb = x[2 * R + 1][c] >> (8 * h);
            uint32_t a0, a1, a2, a3;
            if constexpr (kFp16Mma) {
              const __half2 lo = *reinterpret_cast<const __half2*>(&off_lo);
              const __half2 hi = *reinterpret_cast<const __half2*>(&off_hi);
              uint32_t p0 = gv_lop(xa, 0x000F000Fu, magic);
              uint32_t p1 = gv_lop(xb, 0x000F000Fu, magic);
              uint32_t p2 = gv_lop(xa, 0x00F000F0u, magic);
              uint32_t p3 = gv_lop(xb, 0x00F000F0u, magic);
              __half2 r0 = __hsub2(*reinterpret_cast<__half2*>(&p0), lo);
              __half2 r1 = __hsub2(*reinterpret_cast<__half2*>(&p1), lo);
              __half2 r2 = __hsub2(*reinterpret_cast<__half2*>(&p2), hi);
              __half2 r3 = __hsub2(*reinterpret_cast<__half2*>(&p3), hi);
              a0 = *reinterpret_cast<uint32_t*>(&r0);
              a1 = *reinterpret_cast<uint32_t*>(&r1);
              a2 = *reinterpret_cast<uint32_t*>(&r2);
              a3 = *reinterpret_cast<uint32_t*>(&r3);
            } else {
              a0 = gv_lop(xa, 0x000F000Fu, magic);
              a1 = gv_lop(xb, 0x000F000Fu, magic);
              a2 = gv_lop(xa >> 4, 0x000F000Fu, magic);
              a3 = gv_lop(xb >> 4, 0x000F000Fu, magic);
            }
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              const uint32_t b0 = h ? v[j].z : v[j].x;
              const uint32_t b1 = h ? v[j].w : v[j].y;
              gv_mma<kFp16Mma>(acc[h % H2][R][j], a0, a1, a2, a3, b0, b1);
            }
          }
        if (need_sum) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < NJ; ++j)
              gv_mma<kFp16Mma>(fsum[j], one_lo, one_lo, one_hi, one_hi, h ? v[j].z : v[j].x,
                               h ? v[j].w : v[j].y);
        }
      }
      if (!pc) {  // the group's scale (and zero-point) rows
        const uint8_t* czp = cz + s * 512;
#pragma unroll
        for (int q = 0; q < 2 * RP; ++q) {
          const int row = Cols * w + 8 * q + g;
          if (MODE == kW4A8) {
            isq[q] = args.scales ? static_cast<int>(reinterpret_cast<const int8_t*>(czp)[row]) : 1;
          } else {
            sq[q] = gv_f32(reinterpret_cast<const T16*>(czp)[row]);
            const float z = args.zeros ? gv_f32(reinterpret_cast<const T16*>(czp + 256)[row]) : 0.f;
            cq[q] = kFp16Mma ? z : fmaf(mb, sq[q], z);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // fold at the end of a scale group / exact run, and of the K range
      if (--fleft == 0) fleft = fold_blocks;
      if (kb + 1 == kb1 || fleft == fold_blocks) {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
          for (int R = 0; R < RP; ++R)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = 2 * R + (e >> 1);
              const float a = H2 == 2 ? acc[0][R][j][e] + acc[H2 - 1][R][j][e] : acc[0][R][j][e];
#pragma unroll
              for (int h = 0; h < H2; ++h) acc[h][R][j][e] = 0.f;
              if (MODE == kW4A8) {
                const int blk = __float2int_rn(a);  // exact: sum of a * (q - bias)
                ires[R][j][e] += pc ? blk : isq[q] * blk;
              } else {
                res[R][j][e] = fmaf(sq[q], a, fmaf(-cq[q], fsum[j][e & 1], res[R][j][e]));
              }
            }
#pragma unroll
        for (int j = 0; j < NJ; ++j) fsum[j][0] = fsum[j][1] = fsum[j][2] = fsum[j][3] = 0.f;
      }
    }
    (void)ok;
    // ---- this CTA's sums of its K range: the output (C == 1), or the
    // partial-sum tile of the cluster reduction
    if (C == 1) {
#pragma unroll
      for (int R = 0; R < RP; ++R)
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t m = j * 8 + 2 * t + (e & 1);
            const int64_t n = n0 + Cols * w + 16 * R + g + 8 * (e >> 1);
            if (m < M && n < N) store_out<MODE>(args, m, n, res[R][j][e], ires[R][j][e]);
          }
    } else {
#pragma unroll
      for (int R = 0; R < RP; ++R)
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = j * 8 + 2 * t + (e & 1);
            const int col = Cols * w + 16 * R + g + 8 * (e >> 1);
            red[row * kTileN + col] = MODE == kW4A8 ? static_cast<uint32_t>(ires[R][j][e])
                                                    : __float_as_uint(res[R][j][e]);
          }
    }
  }
  if (C == 1) return;

  // ---- cluster reduction: CTA `rank` owns columns [c_lo, c_hi) of the tile
  cluster_sync();
  {
    const int c_lo = rank * kTileN / C, c_hi = (rank + 1) * kTileN / C;
    const int nc = c_hi - c_lo;
    const int rows = static_cast<int>(M < 8 * NJ ? M : 8 * NJ);
    const uint32_t red0 = smem_addr(red);
    for (int i = threadIdx.x; i < rows * nc; i += GvShape<NJ>::Threads) {
      const int m = i / nc, col = c_lo + (i - m * nc);
      const int64_t n = n0 + col;
      const uint32_t local = red0 + static_cast<uint32_t>(m * kTileN + col) * 4;
      uint32_t parts[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q < C) parts[q] = ld_dsmem(dsmem_addr(local, static_cast<uint32_t>(q)));
      if (n >= N) continue;
      if (MODE == kW4A8) {
        int32_t a = 0;
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (q < C) a += static_cast<int32_t>(parts[q]);
        store_out<MODE>(args, m, n, 0.f, a);
      } else {
        float a = __uint_as_float(parts[0]);
#pragma unroll
        for (int q = 1; q < 16; ++q)
          if (q < C) a += __uint_as_float(parts[q]);
        store_out<MODE>(args, m, n, a, 0);
      }
    }
  }
  cluster_sync();  // every CTA's partial sums stay readable until all are read
}

namespace {
template <int MODE, int NJ>
const void* gv_fn() {
  return reinterpret_cast<const void*>(&gv_gemm_kernel<MODE, NJ>);
}
template <int NJ>
const void* gv_select_nj(int mode) {
  switch (mode) {
    case kW4A16_F16: return gv_fn<kW4A16_F16, NJ>();
    case kW4A16_BF16: return gv_fn<kW4A16_BF16, NJ>();
    case kW4A8F8: return gv_fn<kW4A8F8, NJ>();
    default: return gv_fn<kW4A8, NJ>();
  }
}
const void* gv_select(int mode, int nj) {
  return nj == 1 ? gv_select_nj<1>(mode) : nj == 2 ? gv_select_nj<2>(mode) : gv_select_nj<4>(mode);
}
}  // namespace

int gv_threads(int nj) { return nj >= 4 ? GvShape<4>::Threads : GvShape<1>::Threads; }

// Clusters of C CTAs that can be resident at once; -1 when it cannot be
// determined (no device).
int gv_max_clusters(int mode, int nj, int C, size_t smem) {
  const void* fn = gv_select(mode, nj);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (C > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                   cudaSuccess) {
    cudaGetLastError();
    return 0;  // clusters above 8 CTAs are not available
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(gv_threads(nj));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gv(const GvPlan& plan, const CUtensorMap& amap, const TcArgs& args,
                      cudaStream_t s) {
  const void* fn = gv_select(plan.mode, plan.nj);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan.smem_bytes));
  if (e != cudaSuccess) return e;
  if (plan.cluster > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = plan.cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(gv_threads(plan.nj));
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void* params[3] = {const_cast<CUtensorMap*>(&amap), const_cast<GvPlan*>(&plan),
                     const_cast<TcArgs*>(&args)};
  return cudaLaunchKernelExC(&cfg, fn, params);
}

}  // namespace w4
