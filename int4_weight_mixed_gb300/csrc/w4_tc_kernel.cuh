#pragma once
// w4_tc_kernel.cuh — the tensor-core schedule of the 4-bit-weight GEMM for
// sm_103a: kernel template and its launcher, included by w4_tc.cu (one MMA
// issuer) and w4_tc2.cu (two alternating issuers), so that each kernel
// variant is compiled in a translation unit of its own.
//
// Orientation: the weight tile is the 128-row UMMA "A" operand and the
// activations are the UMMA "B" operand, so each CTA computes
//   D[n, m] = sum_k w_hat[k, n] * a[m, k]      (n: 128 weight columns,
//                                               m: BM activation rows)
// which is the transposed statement of out = a x w_hat (the Machete Readme,
// "Overview", writes the weight on the left of "@ a").
//
// Data flow per pipeline stage (nsub = 1, 2 or 4 blocks of 64 K; the
// stage is sized so that every stage moves >= 8 KB of nibbles for skinny
// tiles, because each stage costs a producer thread a few hundred cycles
// whatever its size):
//   weight producer : one bulk copy of the stage's prepacked nibbles + one
//                   TMA box each of scale / zero-point rows
//   activation producer : one 3-D TMA box of the stage's activations
//                   (128B-swizzled, K-major)
//   16 converter warps (four groups, each converting every fourth stage) :
//                   nibbles -> 16-bit weights in registers, one fused
//                   multiply-add per pair with the scale and pre-scaled
//                   zero-point (Machete Readme "Overview" NOTE), stored
//                   straight into tensor memory (tcgen05.st): dequantized
//                   weights never touch shared memory
//   MMA thread(s) : 4 * nsub tcgen05.mma (K = 16) with A from tensor memory
//                   and B from shared memory, fp32 accumulator in tensor
//                   memory; one commit per stage releases the stage (two
//                   threads alternate by MMA group in the MMA2 variant)
//   epilogue      : converter warps drain the accumulator (tcgen05.ld),
//                   convert / scale and store, or write split-K partials and
//                   let the last arriving warp of each sub-tile add them.
// Warps 0-15 are the converters (warpgroups 0-3); the weight producer, the
// MMA thread, the activation producer and the second MMA thread are warps
// 16-19 (warpgroup 4).
//
// W4A8 (pytorch/ao PR #1113 "support W4A8 Marlin kernel") runs on the same
// bf16 tensor cores: int8 activations and int4 (x int8 group scale)
// weights are exact in bf16, their products are exact in fp32, and the
// accumulator is drained into an int32 running sum before any partial sum
// can exceed 2^24, so the int32 result is exact.  The running sum sits in
// tensor memory beside the accumulator for tiles of up to 128 rows, and in a
// per-CTA global scratch for 256-row tiles (whose accumulator and converted
// stages fill tensor memory).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "w4_epilogue.cuh"
#include "w4_internal.h"
#include "w4_ptx.cuh"

// Converter warpgroups at kTcConvRegs registers and the fifth warpgroup at
// kTcOtherRegs (setmaxnreg at kernel start), or the launch's even split.
#ifndef W4_TC_REGSPLIT
#define W4_TC_REGSPLIT (PAIR || (MODE != kW4A8 && !MMA2))
#endif

namespace w4 {

namespace {

struct Unit {
  int tile;
  int kb0, kb1;
  int nslots;   // units contributing to this tile
  int cfirst;   // first contributing CTA (stream-K)
  int seg;      // index of this tile among the CTA's segments (stream-K)
  int split;    // K split of this unit (split-K)
};

struct Work {
  int64_t T, G, kb;    // G: CTAs, or CTA pairs (the unit of work distribution)
  int64_t me;          // this CTA's (or pair's) index among the G
  int64_t begin, end;  // stream-K range of this CTA (pair)
  int64_t first_tile;
};

__device__ __forceinline__ int64_t sk_start(int64_t c, int64_t T, int64_t G) { return div_nn(c * T, G); }

// Stream-K: the CTA that owns linear iteration i.
__device__ __forceinline__ int64_t sk_owner(int64_t i, int64_t T, int64_t G) {
  return div_nn((i + 1) * G - 1, T);
}

// u-th unit of this CTA; false when there is none.
__device__ bool next_unit(const TcPlan& p, const Work& w, int u, Unit& out) {
  if (p.decomp == kSplitK) {
    // units (tile, split), c, c+G, ...: split j covers stages
    // [j*kb/ks, (j+1)*kb/ks) of its tile
    const int64_t v = w.me + static_cast<int64_t>(u) * w.G;
    if (v >= static_cast<int64_t>(p.tiles) * p.ksplit) return false;
    const int t = static_cast<int>(div_nn(v, p.ksplit)), j = static_cast<int>(v - static_cast<int64_t>(t) * p.ksplit);
    out.tile = t;
    out.split = j;
    out.kb0 = static_cast<int>(div_nn(static_cast<int64_t>(j) * p.kb_total, p.ksplit));
    out.kb1 = static_cast<int>(div_nn(static_cast<int64_t>(j + 1) * p.kb_total, p.ksplit));
    out.nslots = p.ksplit;
    out.cfirst = 0;
    out.seg = 0;
    return true;
  }
  if (p.decomp == kDataParallel) {
    int64_t t = w.me + static_cast<int64_t>(u) * w.G;
    if (t >= p.tiles) return false;
    out.tile = static_cast<int>(t);
    out.kb0 = 0;
    out.kb1 = p.kb_total;
    out.nslots = 1;
    out.cfirst = static_cast<int>(w.me);
    out.seg = 0;
    out.split = 0;
    return true;
  }
  int64_t t = w.first_tile + u;
  int64_t lo = t * w.kb, hi = lo + w.kb;
  if (lo < w.begin) lo = w.begin;
  if (hi > w.end) hi = w.end;
  if (lo >= hi) return false;
  out.tile = static_cast<int>(t);
  out.kb0 = static_cast<int>(lo - t * w.kb);
  out.kb1 = static_cast<int>(hi - t * w.kb);
  int64_t cf = sk_owner(t * w.kb, w.T, w.G);
  int64_t cl = sk_owner((t + 1) * w.kb - 1, w.T, w.G);
  out.cfirst = static_cast<int>(cf);
  out.nslots = static_cast<int>(cl - cf + 1);
  out.seg = u;
  out.split = 0;
  return true;
}

// Partial-sum slot of contributor sl (0-based, in K order) of the unit's tile.
__device__ __forceinline__ size_t slot_index(const TcPlan& p, const Work& w, const Unit& u,
                                             int sl) {
  if (p.decomp == kSplitK) return static_cast<size_t>(u.tile) * p.ksplit + sl;
  const int64_t cpr = u.cfirst + sl;
  const int64_t seg = u.tile - div_nn(sk_start(cpr, w.T, w.G), w.kb);
  return static_cast<size_t>(cpr) * p.max_segs + seg;
}
__device__ __forceinline__ size_t own_slot(const TcPlan& p, const Work& w, const Unit& u) {
  if (p.decomp == kSplitK) return static_cast<size_t>(u.tile) * p.ksplit + u.split;
  return static_cast<size_t>(w.me) * p.max_segs + u.seg;
}

// Tile -> (m_tile, n_tile), grouped raster: runs of up to 8 m-tiles share
// each weight tile while it is in L2.
__device__ __forceinline__ void tile_coords(const TcPlan& p, int t, int& mt, int& nt) {
  int gm_full = p.m_tiles < 8 ? p.m_tiles : 8;
  int group = t / (gm_full * p.n_tiles);
  int local = t - group * gm_full * p.n_tiles;
  int gm = p.m_tiles - group * gm_full;
  if (gm > gm_full) gm = gm_full;
  mt = group * gm_full + local % gm;
  nt = local / gm;
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

template <typename T2>
__device__ __forceinline__ T2 as_t2(uint32_t x) {
  return *reinterpret_cast<T2*>(&x);
}
template <typename T2>
__device__ __forceinline__ uint32_t as_u32(T2 x) {
  return *reinterpret_cast<uint32_t*>(&x);
}

// Dequantize the 32 K-values of one 16-byte chunk (4 words, ExLlama order)
// into 16 packed pairs.  Pair p of word x holds (k0+2p, k0+2p+1) at bits
// (4p, 16+4p).  OR-ing a nibble into the mantissa of the "magic" constant
// gives magic+q exactly; subtracting magic+bias is exact; the FMA with the
// scale and negated zero-point rounds once.
template <int MODE>
__device__ __forceinline__ void convert_chunk(const uint4& wv, uint32_t s2u, uint32_t nz2u,
                                              bool has_z, bool has_s, int wbias,
                                              uint32_t (&v)[16]) {
  const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
  if constexpr (MODE == kW4A16_F16) {
    const __half2 off = __half2half2(__int2half_rn(1024 + wbias));
    const __half2 s2 = as_t2<__half2>(s2u), nz2 = as_t2<__half2>(nz2u);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        __half2 h = as_t2<__half2>(lop_and_or(wd[i] >> (4 * p), 0x000F000Fu, 0x64006400u));
        __half2 q = __hsub2(h, off);
        v[4 * i + p] = as_u32(has_z ? __hfma2(q, s2, nz2) : __hmul2(q, s2));
      }
  } else {
    const __nv_bfloat162 off = __bfloat162bfloat162(__int2bfloat16_rn(128 + wbias));
    const __nv_bfloat162 s2 = as_t2<__nv_bfloat162>(s2u), nz2 = as_t2<__nv_bfloat162>(nz2u);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        __nv_bfloat162 h =
            as_t2<__nv_bfloat162>(lop_and_or(wd[i] >> (4 * p), 0x000F000Fu, 0x43004300u));
        __nv_bfloat162 q = __hsub2(h, off);
        if constexpr (MODE == kW4A8) {
          v[4 * i + p] = as_u32(has_s ? __hmul2(q, s2) : q);
        } else {
          v[4 * i + p] = as_u32(has_z ? __hfma2(q, s2, nz2) : __hmul2(q, s2));
        }
      }
  }
}

// E4M3 weights for W4A8 with fp8 activations: the 32 K-values of one
// 16-byte chunk as eight 32-bit tensor-memory columns of four E4M3 bytes in K
// order.  Each nibble pair becomes the exact fp16 pair (q - bias) by the
// exponent-bias trick, which one conversion turns into two E4M3 bytes
// (exact: every value -8..7 is an E4M3 value); two byte pairs make a column.
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}
__device__ __forceinline__ void convert_chunk_f8(const uint4& wv, int wbias, uint32_t* v) {
  const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
  const __half2 off = __half2half2(__int2half_rn(1024 + wbias));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint16_t e[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const __half2 q = __hsub2(as_t2<__half2>(lop_and_or(wd[i] >> (4 * p), 0x000F000Fu,
                                                          0x64006400u)),
                                off);
      e[p] = f16x2_to_e4m3x2(as_u32(q));  // K 2p (low byte), 2p + 1
    }
    v[2 * i] = static_cast<uint32_t>(e[0]) | (static_cast<uint32_t>(e[1]) << 16);
    v[2 * i + 1] = static_cast<uint32_t>(e[2]) | (static_cast<uint32_t>(e[3]) << 16);
  }
}

template <typename T>
__device__ __forceinline__ T to_t16(float x);
template <>
__device__ __forceinline__ __half to_t16<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 to_t16<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

struct Smem {
  uint8_t* a;       // stages x nsub x BM x 128 B  (128B-swizzled activation tiles)
  uint8_t* w;       // stages x nsub x 4096 B      (prepacked nibbles)
  uint8_t* s;       // stages x nsub x 256 B       (scale rows, up to nsub groups)
  uint8_t* z;       // stages x nsub x 256 B       (zero-point rows)
  uint64_t* full;   // [kMaxStages]  TMA bytes landed
  uint64_t* empty;  // [kMaxStages]  stage consumed (converter group + MMA commit)
  uint64_t* tfull;  // [kMaxTmemStages] converted weights stored in tensor memory
  uint64_t* dfull;  // accumulator ready for the epilogue
  uint64_t* dempty; // accumulator drained
  uint64_t* fin;    // all MMAs retired (before tensor memory is freed)
  uint64_t* tok;    // [2] MMA issuing turn of thread 0 / 1
  uint32_t* tmem_slot;
  int* abort;
};

}  // namespace

// d (fp32 sums of one W4A8 chunk, exact integers below 2^24) becomes its
// int32 value plus the running sum prev (unless this is the first chunk).
__device__ __forceinline__ void add_chunk_sums(uint32_t (&d)[8], const uint32_t (&prev)[8],
                                               bool first) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t v = static_cast<uint32_t>(__float2int_rn(__uint_as_float(d[k])));
    d[k] = first ? v : v + prev[k];
  }
}

// MMA2: two alternating MMA-issuing threads; a separate instantiation.
// PAIR: a cluster of two CTAs shares every MMA (cta_group::2, M = 256): CTA
// rank r converts weight columns [n0 + 128r, n0 + 128r + 128) of the pair's
// 256-column tile into its own tensor memory and loads activation rows
// [y + BM/2 r, y + BM/2 (r + 1)) of the BM-row tile into its own shared
// memory; rank 0 issues the MMAs, which give each CTA the sums of its 128
// weight columns against all BM rows.  Per SM the MMA work of a stage is
// that of a single CTA, but the activation bytes per stage halve, so twice
// as many stages fit in shared memory.
// LEAN (CTA pairs): the single 128-column weight tile of each CTA is a
// compile-time constant, and the stream-K partial sums use the layout of the
// running sums (each 16-byte access of a warp covering 512 contiguous
// bytes).  Measured (chained launches, N=8192 K=21760): grouped W4A8 7-9%,
// fp8 activations 5% and W4A16 prefill 3-6% faster with it, while the
// per-channel W4A8 pair kernel, whose time is spent in a few long exact
// chunks and the stream-K fix-up, was 3-14% slower in every variant of it
// tried; that one is instantiated without it.
template <int MODE, bool MMA2, bool PAIR = false, bool LEAN = false>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap amap,
                   const __grid_constant__ CUtensorMap smap,
                   const __grid_constant__ CUtensorMap zmap, const TcPlan p, const TcArgs args) {
  using T16 = typename std::conditional<MODE == kW4A16_F16, __half, __nv_bfloat16>::type;
  // W4A8 with fp8 activations: K blocks of 128 E4M3 values (one 128-byte
  // activation row, 8 KB of nibbles per 128-column tile) on kind::f8f6f4;
  // otherwise blocks of 64 16-bit values (4 KB of nibbles) on kind::f16
  constexpr bool F8 = MODE == kW4A8F8;
  constexpr int BK = F8 ? 128 : kStageK;
  constexpr uint32_t WB = F8 ? 8192u : 4096u;
  constexpr int CPB = BK / kChunkK;  // 32-K chunks per block
  constexpr int NCTA = PAIR ? 2 : 1;
  if constexpr (PAIR) {
    // launched without its two-CTA clusters: nothing may run
    if (cluster_size() != 2) {
      if (threadIdx.x == 0) atomicExch(args.status, 4 /* W4_ERR_CUDA */);
      return;
    }
  }
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  // converter groups visit only their own stages (see the converter loop)
  constexpr bool kOwnStages = PAIR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages, BM = p.bm, NS = p.nsub, TS = p.tstages, NT = LEAN ? 1 : p.nt;
  const int BMc = BM / NCTA;  // activation rows held by this CTA
  const uint32_t a_sub = static_cast<uint32_t>(BMc) * 128;  // bytes of one 64-K activation tile
  Smem sm;
  sm.a = base;
  sm.w = sm.a + static_cast<size_t>(S) * NS * a_sub;             // [S][NT][NS][4096]
  sm.s = sm.w + static_cast<size_t>(S) * NT * NS * WB;            // [S][NT][NS * 256]
  sm.z = sm.s + static_cast<size_t>(S) * NT * NS * 256;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.z + static_cast<size_t>(S) * NT * NS * 256);
  sm.full = bars;
  sm.empty = bars + kMaxStages;
  sm.tfull = bars + 2 * kMaxStages;
  sm.dfull = sm.tfull + kMaxTmemStages;
  sm.dempty = sm.dfull + 1;
  sm.fin = sm.dempty + 1;
  sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.fin + 1);
  sm.abort = reinterpret_cast<int*>(sm.tmem_slot + 1);
  sm.tok = sm.fin + 2;  // after the slot and abort words (8-byte aligned)
  volatile int* abort = sm.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&sm.full[i], 1);  // the producer thread of the stage's parity
      mbar_init(&sm.empty[i], 4 + 1);  // one converter group + the MMA commit
    }
    // tfull / dempty: the converter warps of both CTAs of a pair arrive on
    // rank 0's (the other CTA's copies stay unused)
    for (int i = 0; i < TS; ++i) mbar_init(&sm.tfull[i], 4 * NCTA);
    mbar_init(sm.dfull, 1);
    mbar_init(sm.dempty, kConvWarps * NCTA);
    mbar_init(sm.fin, MMA2 ? 2 : 1);  // one commit per MMA issuing thread
    if constexpr (MMA2) {
      mbar_init(&sm.tok[0], 1);
      mbar_init(&sm.tok[1], 1);
    }
    *sm.abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&amap);
    if (args.scales) prefetch_tensormap(&smap);
    if (args.zeros) prefetch_tensormap(&zmap);
  }
  if (warp == kProdWarp) {
    if constexpr (PAIR) {
      tmem_alloc_pair(sm.tmem_slot, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(sm.tmem_slot, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers initialised
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;
  // rank 0's tfull / dempty, as seen from this CTA
  const uint32_t tfull_c = PAIR ? peer_addr(smem_addr(sm.tfull), 0) : smem_addr(sm.tfull);
  const uint32_t dempty_c = PAIR ? peer_addr(smem_addr(sm.dempty), 0) : smem_addr(sm.dempty);


  Work wk;
  wk.kb = p.kb_total;
  wk.T = static_cast<int64_t>(p.tiles) * p.kb_total;
  wk.G = p.grid / NCTA;
  wk.me = blockIdx.x / NCTA;
  wk.begin = sk_start(wk.me, wk.T, wk.G);
  wk.end = sk_start(wk.me + 1, wk.T, wk.G);
  wk.first_tile = div_nn(wk.begin, wk.kb);

  const int64_t M = args.M, N = args.N, K = args.K;
  const int gsz = static_cast<int>(args.group_size);
  const int sub_per_group = gsz / BK;  // K blocks per scale group
  // A stage lies inside one scale group (sub_per_group >= NS) or covers whole
  // groups of 1 or 2 blocks (the plan guarantees one or the other): the group
  // of block qq of a stage is the stage's first group + (qq >> grow_shift).
  const bool stage_in_group = sub_per_group >= NS;
  const int grow_shift = sub_per_group >= 2 ? 1 : 0;
  const int esz = MODE == kW4A8 ? 1 : 2;

  if (warp >= kConvWarps) {
  // W4A16 with one MMA issuer: the fifth warpgroup (producers, MMA) gives
  // registers to the converters, whose scale / zero-point FMAs otherwise
  // spill (the other kernels keep the even split: measured faster)
  if constexpr (W4_TC_REGSPLIT)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTcOtherRegs));
  if (warp == kProdWarp || warp == kActWarp) {
    // ----------------------------------------------------------- producers
    // Two single-thread producers take alternate stages; for each of its
    // stages a producer issues the bulk copy of the stage's nibbles, the
    // scale / zero-point boxes and the activation tile(s), with one expect-tx
    // on the stage's full barrier.
    if (lane == 0) {
      const bool wprod = warp == kProdWarp;
      // W4A8: the activations come from the staging grid this one may have
      // been launched beside (programmatic dependent launch); wait for it
      // Each of the two threads issues every copy of alternate stages (stage
      // it goes to the thread with it % 2 == pid), stepping two stages at a
      // time: one thread issuing the weights of every stage was the stage
      // rate's limit (its dependent instruction chain per stage, on a
      // sub-partition shared with four converter warps, took as long as the
      // stage's MMAs).
      const uint32_t pid = wprod ? 0u : 1u;
      bool waited = false;  // W4A8: the staging grid this one may overlap
      uint32_t n_issued = 0, last_it = 0;  // stages this thread issued, the last one
      uint32_t it_u = 0;    // stage index of the unit's first stage
      bool ok = true;
      Unit u;
      const uint32_t a0 = smem_addr(sm.a), w0 = smem_addr(sm.w);
      const uint32_t s0 = smem_addr(sm.s), z0 = smem_addr(sm.z);
      const uint32_t full0 = smem_addr(sm.full);
      const uint32_t sc_bytes = args.scales ? static_cast<uint32_t>(128 * p.gps * esz) : 0;
      const uint32_t zp_bytes = args.zeros ? static_cast<uint32_t>(128 * p.gps * 2) : 0;
      for (int ui = 0; ok && next_unit(p, wk, ui, u); ++ui) {
        int mt, nt;
        tile_coords(p, u.tile, mt, nt);
        const int wt0 = (nt * NCTA + static_cast<int>(rank)) * NT;  // first weight tile of this CTA
        const int32_t n0 = wt0 * kTileN;           // first weight column of the CTA tile
        const int32_t y = mt * BM + static_cast<int>(rank) * BMc;
        int ntv = p.n128 - wt0;                     // weight tiles that exist (ragged N)
        if (ntv > NT) ntv = NT;
        if (ntv < 0) ntv = 0;
        const int64_t tile_stride = (K / kChunkK) * kTileN * 16;  // bytes between weight tiles
        // this thread's first stage of the unit, and its ring slot / phase
        const int kbf = u.kb0 + static_cast<int>((pid + 2u - (it_u & 1u)) & 1u);
        uint32_t it = it_u + static_cast<uint32_t>(kbf - u.kb0);
        uint32_t s = it % S, ph = (it / S) & 1u;
        const uint8_t* wsrc =
            args.b_packed +
            ((static_cast<int64_t>(wt0) * (K / kChunkK) + static_cast<int64_t>(kbf) * NS * CPB) *
             kTileN) * 16;
        // scale group of the stage, kept without division per stage
        int gcur = kbf * NS / sub_per_group;
        int gleft = sub_per_group - (kbf * NS) % sub_per_group;
        for (int kb = kbf; kb < u.kb1; kb += 2, it += 2) {
          if (!mbar_wait<true>(&sm.empty[s], ph ^ 1, abort, args.status)) { ok = false; break; }
          const int k64_0 = kb * NS;
          const int nv = p.k64 - k64_0 < NS ? p.k64 - k64_0 : NS;  // valid 64-K blocks
          const uint32_t fb = full0 + s * 8;
          const uint32_t abytes = p.a3d ? NS * a_sub : nv * a_sub;
          mbar_arrive_expect_tx_a(fb, ntv * nv * WB + NT * (sc_bytes + zp_bytes) + abytes);
          for (int t = 0; t < ntv; ++t)
            bulk_g2s_a(w0 + (s * NT + t) * NS * WB, wsrc + t * tile_stride, nv * WB, fb);
          if (sc_bytes || zp_bytes) {
            const int g0 = gcur;
            for (int t = 0; t < NT; ++t) {
              if (sc_bytes)
                tma_load_2d_a(s0 + (s * NT + t) * NS * 256, &smap, n0 + t * kTileN, g0, fb);
              if (zp_bytes)
                tma_load_2d_a(z0 + (s * NT + t) * NS * 256, &zmap, n0 + t * kTileN, g0, fb);
            }
          }
          // W4A8: the activations come from the staging grid this one may
          // have been launched beside (programmatic dependent launch); the
          // weights of the first stage are already on their way
          if (!waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
          }
          if (p.a3d) {
            tma_load_3d_a(a0 + s * NS * a_sub, &amap, 0, y, k64_0, fb);
          } else {
            for (int j = 0; j < nv; ++j)
              tma_load_2d_a(a0 + (s * NS + j) * a_sub, &amap, (k64_0 + j) * BK, y, fb);
          }
          ++n_issued;
          last_it = it;
          wsrc += 2 * NS * WB;
          if (stage_in_group) {
            gleft -= 2 * NS;
            while (gleft <= 0) {
              ++gcur;
              gleft += sub_per_group;
            }
          } else {
            gcur += 2 * p.gps;
          }
          s += 2;
          if (s >= static_cast<uint32_t>(S)) {
            s -= S;
            ph ^= 1;
          }
        }
        it_u += static_cast<uint32_t>(u.kb1 - u.kb0);
      }
      // Let every copy this thread issued land before the CTA can exit: its
      // stages among the last S of the whole sequence, the final users of
      // their slots (an earlier stage's slot may have been refilled, and with
      // an odd S by the other thread, so a parity wait on it would be
      // ambiguous).  After an abort: its own last S stages.
      const uint32_t end = ok ? it_u : last_it + 1;
      if (n_issued > 0)
        for (uint32_t j = (end > static_cast<uint32_t>(S) ? end - S : 0); j < end; ++j) {
          if ((j & 1u) != pid || j > last_it) continue;
          volatile int no_abort = 0;
          mbar_wait<true>(&sm.full[j % S], (j / S) & 1, &no_abort, args.status);
        }
    }
  } else if (warp == kMmaWarp || warp == kMma2Warp) {
    // ----------------------------------------------------------------- MMA
    // With MMA2, two issuing threads take turns by MMA group (one stage, or
    // two one-block stages): the issuing thread is held inside each
    // tcgen05.mma for about its execution time, so one thread's barrier waits
    // and bookkeeping run while the other's MMAs keep the tensor pipe busy.  A
    // group is issued only after the previous one (token barrier between
    // tcgen05 fences), so the pipe receives the groups in K order, and the
    // issuer of a chunk's last group alone signals the accumulator ready: its
    // MMAs accumulate after all earlier ones.  Without MMA2, the MMA warp
    // alone issues every group (the loop right below).
    if constexpr (!MMA2) {
    if (lane == 0 && warp == kMmaWarp && rank != 0) {
      // a pair's MMAs are issued by rank 0: wait for their last commit, so
      // that this CTA's tensor and shared memory outlive them
      volatile int no_abort = 0;
      mbar_wait<true>(sm.fin, 0, &no_abort, args.status);
    } else if (lane == 0 && warp == kMmaWarp) {
      const uint32_t idesc = idesc_f16_m(MODE == kW4A16_BF16 || MODE == kW4A8 ? 1u : 0u,
                                         static_cast<uint32_t>(BM), PAIR ? 256u : 128u);
      const uint64_t desc0 = sw128_kmajor_desc(smem_addr(sm.a));
      const uint32_t sub16 = a_sub / 16;  // descriptor address units per activation tile
      uint32_t s = 0, ph = 0, ts = 0, tph = 0, ev = 0;
      bool ok = true;
      Unit u;
      auto wait_x = [&](uint64_t* bar, uint32_t par) {
        return mbar_wait<true>(bar, par, abort, args.status);
      };
      auto commit = [&](uint64_t* bar) {
        if constexpr (PAIR) mma_commit_pair(bar);
        else mma_commit(bar);
      };
      for (int ui = 0; ok && next_unit(p, wk, ui, u); ++ui) {
        bool chunk_start = true;
        const int nkb = u.kb1 - u.kb0;
        // stages of the current exact chunk (W4A8) or of the unit still to go
        const int chunk_len = MODE == kW4A8 ? p.chunk_stages : nkb;
        int left = 0;
        auto advance = [&]() {
          if (++s == static_cast<uint32_t>(S)) {
            s = 0;
            ph ^= 1;
          }
          if (++ts == static_cast<uint32_t>(TS)) {
            ts = 0;
            tph ^= 1;
          }
        };
        for (int j = 0; j < nkb;) {
          if (chunk_start) {
            if (ev > 0 && !wait_x(sm.dempty, (ev - 1) & 1)) {
              ok = false;
              break;
            }
            left = chunk_len < nkb - j ? chunk_len : nkb - j;
          }
          // One-block stages go to the tensor pipe two at a time (eight MMAs
          // per group) when both belong to the same exact chunk.
          const bool pair = NS == 1 && NT == 1 && TS >= 2 && left >= 2;
          // The converter group arrives on tfull only after it observed the
          // stage's full barrier, so tfull also orders the activation tile
          // (of both CTAs of a pair).
          if (!wait_x(&sm.tfull[ts], tph)) {
            ok = false;
            break;
          }
          const uint32_t s1 = s, ts1 = ts;
          uint32_t s2 = s + 1, ts2 = ts + 1, tph2 = tph;
          if (s2 == static_cast<uint32_t>(S)) s2 = 0;
          if (ts2 == static_cast<uint32_t>(TS)) {
            ts2 = 0;
            tph2 ^= 1;
          }
          if (pair && !wait_x(&sm.tfull[ts2], tph2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool two_blocks = NS == 2 && NT == 1 && p.k64 - (u.kb0 + j) * NS >= 2;
          if (pair || two_blocks) {
            // eight MMAs: two stages of one 64-K block, or one stage of two
            uint32_t a8[8];
            uint64_t b8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int half = i >> 2, kk = i & 3;
              if (pair) {
                a8[i] = tmem + p.acol + (half ? ts2 : ts1) * 32 + 8 * kk;
                b8[i] = desc0 + (half ? s2 : s1) * sub16 + 2 * kk;
              } else {
                a8[i] = tmem + p.acol + ts1 * 64 + 32 * half + 8 * kk;
                b8[i] = desc0 + s1 * 2 * sub16 + half * sub16 + 2 * kk;
              }
            }
            if (MODE == kW4A8 && pair) {
              // W4A8: the first stage's shared-memory slot is released as soon
              // as its own four MMAs retire (measured 3% faster at 256-row
              // tiles; W4A16 measured slower with the extra commit)
              if constexpr (PAIR) {
                mma_pair_4<F8>(tmem, a8, b8, idesc, chunk_start ? 0u : 1u);
                commit(&sm.empty[s1]);
                mma_pair_4<F8>(tmem, a8 + 4, b8 + 4, idesc, 1u);
              } else {
                mma_ts_4<F8>(tmem, a8, b8, idesc, chunk_start ? 0u : 1u);
                commit(&sm.empty[s1]);
                mma_ts_4<F8>(tmem, a8 + 4, b8 + 4, idesc, 1u);
              }
            } else {
              if constexpr (PAIR) mma_pair_8<F8>(tmem, a8, b8, idesc, chunk_start ? 0u : 1u);
              else mma_ts_8<F8>(tmem, a8, b8, idesc, chunk_start ? 0u : 1u);
            }
          } else if constexpr (PAIR) {
            // a stage of one K block (NS = 1, or the last, one-block stage of
            // NS = 2; the pair kernel has NT = 1)
            uint32_t a4[4];
            uint64_t b4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              a4[i] = tmem + p.acol + ts * NS * 32 + 8 * i;
              b4[i] = desc0 + s * NS * sub16 + 2 * i;
            }
            mma_pair_4<F8>(tmem, a4, b4, idesc, chunk_start ? 0u : 1u);
          } else {
            const int k64_0 = (u.kb0 + j) * NS;
            const int nv = p.k64 - k64_0 < NS ? p.k64 - k64_0 : NS;
            for (int t = 0; t < NT; ++t) {
              const uint32_t dcol = tmem + t * BM;
              const uint32_t acol = tmem + p.acol + (ts * NT + t) * NS * 32;
              const uint64_t dsc = desc0 + s * NS * sub16;
              if (nv == 4) {
                mma_ts_stage16<F8>(dcol, acol, dsc, sub16, idesc, chunk_start ? 0u : 1u);
              } else {
                mma_ts_stage<F8>(dcol, acol, dsc, idesc, chunk_start ? 0u : 1u);
                for (int q = 1; q < nv; ++q)
                  mma_ts_stage<F8>(dcol, acol + q * 32, dsc + q * sub16, idesc, 1u);
              }
            }
          }
          if (!(MODE == kW4A8 && pair)) commit(&sm.empty[s1]);
          advance();
          if (pair) {
            commit(&sm.empty[s2]);
            advance();
          }
          const int used = pair ? 2 : 1;
          j += used;
          left -= used;
          chunk_start = false;
          if (left == 0) {
            commit(sm.dfull);
            ++ev;
            chunk_start = true;
          }
        }
      }
      // All issued MMAs complete before tensor memory is released.
      commit(sm.fin);
      volatile int no_abort = 0;
      mbar_wait<true>(sm.fin, 0, &no_abort, args.status);
    }
    } else {
    if (lane == 0 && rank != 0) {
      // a pair's MMAs are issued by rank 0: wait for their last commits
      if (warp == kMmaWarp) {
        volatile int no_abort = 0;
        mbar_wait<true>(sm.fin, 0, &no_abort, args.status);
      }
    } else if (lane == 0) {
      const uint32_t me = warp == kMmaWarp ? 0u : 1u;  // issues the groups g with g % 2 == me
      const uint32_t idesc = idesc_f16_m(MODE == kW4A16_BF16 || MODE == kW4A8 ? 1u : 0u,
                                         static_cast<uint32_t>(BM), PAIR ? 256u : 128u);
      auto commit = [&](uint64_t* bar) {
        if constexpr (PAIR) mma_commit_pair(bar);
        else mma_commit(bar);
      };
      const uint64_t desc0 = sw128_kmajor_desc(smem_addr(sm.a));
      const uint32_t sub16 = a_sub / 16;  // descriptor address units per activation tile
      uint32_t s = 0, ph = 0, ts = 0, tph = 0, ev = 0, g = 0, tok_ph = 0;
      bool ok = true, issued = false;
      Unit u;
      for (int ui = 0; ok && next_unit(p, wk, ui, u); ++ui) {
        bool chunk_start = true;
        const int nkb = u.kb1 - u.kb0;
        // stages of the current exact chunk (W4A8) or of the unit still to go
        const int chunk_len = MODE == kW4A8 ? p.chunk_stages : nkb;
        int left = 0;
        auto advance = [&]() {
          if (++s == static_cast<uint32_t>(S)) {
            s = 0;
            ph ^= 1;
          }
          if (++ts == static_cast<uint32_t>(TS)) {
            ts = 0;
            tph ^= 1;
          }
        };
        for (int j = 0; j < nkb; ++g) {
          if (chunk_start) left = chunk_len < nkb - j ? chunk_len : nkb - j;
          // One-block stages go to the tensor pipe two at a time (eight MMAs
          // per group) when both belong to the same exact chunk.
          const bool pair = NS == 1 && NT == 1 && TS >= 2 && left >= 2;
          const int used = pair ? 2 : 1;
          const bool chunk_end = left == used;
          if ((g & 1u) == me) {
            if (chunk_start && ev > 0 && !mbar_wait<true>(sm.dempty, (ev - 1) & 1, abort, args.status)) {
              ok = false;
              break;
            }
            // The converter group arrives on tfull only after it observed the
            // stage's full barrier, so tfull also orders the activation tile.
            if (!mbar_wait<true>(&sm.tfull[ts], tph, abort, args.status)) {
              ok = false;
              break;
            }
            const uint32_t s1 = s, ts1 = ts;
            uint32_t s2 = s + 1, ts2 = ts + 1, tph2 = tph;
            if (s2 == static_cast<uint32_t>(S)) s2 = 0;
            if (ts2 == static_cast<uint32_t>(TS)) {
              ts2 = 0;
              tph2 ^= 1;
            }
            if (pair && !mbar_wait<true>(&sm.tfull[ts2], tph2, abort, args.status)) {
              ok = false;
              break;
            }
            // the other thread has issued the previous group (waited last,
            // so that the pipe changes hands with the least delay)
            if (g > 0) {
              if (!mbar_wait<true>(&sm.tok[me], tok_ph, abort, args.status)) {
                ok = false;
                break;
              }
              tok_ph ^= 1;
            }
            tc_fence_after();
            const bool two_blocks = NS == 2 && NT == 1 && p.k64 - (u.kb0 + j) * NS >= 2;
            if (pair || two_blocks) {
              // eight MMAs: two stages of one 64-K block, or one stage of two
              uint32_t a8[8];
              uint64_t b8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int half = i >> 2, kk = i & 3;
                if (pair) {
                  a8[i] = tmem + p.acol + (half ? ts2 : ts1) * 32 + 8 * kk;
                  b8[i] = desc0 + (half ? s2 : s1) * sub16 + 2 * kk;
                } else {
                  a8[i] = tmem + p.acol + ts1 * 64 + 32 * half + 8 * kk;
                  b8[i] = desc0 + s1 * 2 * sub16 + half * sub16 + 2 * kk;
                }
              }
              if constexpr (PAIR) mma_pair_8<F8>(tmem, a8, b8, idesc, chunk_start ? 0u : 1u);
              else mma_ts_8<F8>(tmem, a8, b8, idesc, chunk_start ? 0u : 1u);
            } else if constexpr (PAIR) {
              // a stage of one K block (NS = 1, or the last, one-block stage
              // of NS = 2; the pair kernel has NT = 1)
              uint32_t a4[4];
              uint64_t b4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                a4[i] = tmem + p.acol + ts * NS * 32 + 8 * i;
                b4[i] = desc0 + s * NS * sub16 + 2 * i;
              }
              mma_pair_4<F8>(tmem, a4, b4, idesc, chunk_start ? 0u : 1u);
            } else {
              const int k64_0 = (u.kb0 + j) * NS;
              const int nv = p.k64 - k64_0 < NS ? p.k64 - k64_0 : NS;
              for (int t = 0; t < NT; ++t) {
                const uint32_t dcol = tmem + t * BM;
                const uint32_t acol = tmem + p.acol + (ts * NT + t) * NS * 32;
                const uint64_t dsc = desc0 + s * NS * sub16;
                if (nv == 4) {
                  mma_ts_stage16<F8>(dcol, acol, dsc, sub16, idesc, chunk_start ? 0u : 1u);
                } else {
                  mma_ts_stage<F8>(dcol, acol, dsc, idesc, chunk_start ? 0u : 1u);
                  for (int q = 1; q < nv; ++q)
                    mma_ts_stage<F8>(dcol, acol + q * 32, dsc + q * sub16, idesc, 1u);
                }
              }
            }
            // hand the pipe over, then release the stages (a commit tracks
            // this thread's own MMAs)
            tc_fence_before();
            mbar_arrive(&sm.tok[me ^ 1u]);
            commit(&sm.empty[s1]);
            if (pair) commit(&sm.empty[s2]);
            if (chunk_end) commit(sm.dfull);
            issued = true;
          }
          advance();
          if (pair) advance();
          j += used;
          left -= used;
          chunk_start = false;
          if (left == 0) {
            ++ev;
            chunk_start = true;
          }
        }
      }
      // All issued MMAs complete before tensor memory is released (a thread
      // that issued none arrives directly; in a pair it commits all the
      // same, which reaches both CTAs' barriers at once).
      if (PAIR || issued) commit(sm.fin);
      else mbar_arrive(sm.fin);
      volatile int no_abort = 0;
      mbar_wait<true>(sm.fin, 0, &no_abort, args.status);
    }
    }
  }
  } else {
    if constexpr (W4_TC_REGSPLIT)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTcConvRegs));
    // ----------------------------------------------- converters + epilogue
    const int cw = warp;               // converter warp index 0..kConvWarps-1
    const int grp = cw >> 2;           // group: converts stages it % kConvGroups == grp
    const int q = warp & 3;            // tensor-memory lane quadrant of this warp
    const int r = q * 32 + lane;       // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int nblk = BM / 8;           // 8-column blocks of the accumulator
    uint32_t it_u = 0, ev = 0;  // it_u: the unit's first stage in this CTA's stage sequence
    bool ok = true;
    Unit u;
    for (int ui = 0; ok && next_unit(p, wk, ui, u); ++ui) {
      int mt, nt;
      tile_coords(p, u.tile, mt, nt);
      // first weight column of this CTA's tile; the accumulator covers all BM
      // rows of the (pair's) tile
      const int64_t n0 = (static_cast<int64_t>(nt) * NCTA + rank) * NT * kTileN;
      const int64_t m0 = static_cast<int64_t>(mt) * BM;
      const int nkb = u.kb1 - u.kb0;
      const int chunk_len = MODE == kW4A8 ? p.chunk_stages : nkb;
      bool first_chunk = true;
      // one stage of this group (stage it of the sequence, j of the unit, in
      // shared-memory slot s with phase cph and tensor-memory slot ts; stage
      // it - TS in slot ps with phase pph); false when a wait gave up
      auto conv_stage = [&](int j, uint32_t it, uint32_t s, uint32_t cph, uint32_t ts,
                            uint32_t ps, uint32_t pph) -> bool {
        // The tensor-memory slot first: it is free once the MMA of stage
        // it-TS retired.  MMAs retire in order, so stage it-S (TS < S),
        // the previous user of shared-memory slot s, has then been converted
        // and its copies have landed; only after that is the parity wait on
        // full[s] unambiguous.  (A group converts every kConvGroups-th stage:
        // nothing else orders this group's wait after the landing of stage
        // it-S, which another group converted; were that phase still
        // pending, the parity wait would pass at once.)  The slot wait itself
        // is unambiguous for S >= kConvGroups: this group's previous slot
        // wait (stage it-kConvGroups-TS) already covers stage it-TS-S.
        if (it >= static_cast<uint32_t>(TS)) {
          if (!__all_sync(0xffffffffu, mbar_wait<true>(&sm.empty[ps], pph, abort, args.status))) {
            return false;
          }
        }
        if (!__all_sync(0xffffffffu, mbar_wait<true>(&sm.full[s], cph, abort, args.status))) {
          return false;
        }
        tc_fence_after();
        const int k64_0 = (u.kb0 + j) * NS;
        const int nv = p.k64 - k64_0 < NS ? p.k64 - k64_0 : NS;
        for (int t = 0; t < NT; ++t) {
          const size_t st_idx = static_cast<size_t>(s) * NT + t;
          const uint8_t* wst = sm.w + st_idx * NS * WB;
          const uint8_t* sst = sm.s + st_idx * NS * 256;
          const uint8_t* zst = sm.z + st_idx * NS * 256;
          const uint32_t tcol = tmem + lane_base + p.acol + (ts * NT + t) * NS * 32;
          const bool row_ok = n0 + t * kTileN + r < N;
          for (int qq = 0; qq < nv; ++qq) {
            if constexpr (F8) {
              // four 32-K chunks -> 32 columns of E4M3 bytes (no scales)
              uint32_t v[32];
#pragma unroll
              for (int c = 0; c < 4; ++c)
                convert_chunk_f8(*reinterpret_cast<const uint4*>(wst + qq * WB + c * 2048 + r * 16),
                                 args.wbias, v + 8 * c);
              if (!row_ok) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0;
              }
              tmem_st32(tcol + qq * 32, v);
              continue;
            }
            const uint4 w0 = *reinterpret_cast<const uint4*>(wst + qq * 4096 + r * 16);
            const uint4 w1 = *reinterpret_cast<const uint4*>(wst + qq * 4096 + 2048 + r * 16);
            const int grow = stage_in_group ? 0 : qq >> grow_shift;
            uint32_t s2 = 0, nz2 = 0;
            bool has_s = true;
            if (MODE == kW4A8) {
              has_s = args.scales != nullptr;
              if (has_s) {
                const float sg = static_cast<float>(
                    reinterpret_cast<const int8_t*>(sst + grow * 128)[r]);
                s2 = as_u32(__float2bfloat162_rn(sg));
              }
            } else {
              const uint16_t sv = reinterpret_cast<const uint16_t*>(sst + grow * 256)[r];
              s2 = static_cast<uint32_t>(sv) | (static_cast<uint32_t>(sv) << 16);
              if (args.zeros) {
                const uint16_t zv =
                    reinterpret_cast<const uint16_t*>(zst + grow * 256)[r] ^ 0x8000u;
                nz2 = static_cast<uint32_t>(zv) | (static_cast<uint32_t>(zv) << 16);
              }
            }
            uint32_t v[32];
            uint32_t (&v0)[16] = *reinterpret_cast<uint32_t(*)[16]>(&v[0]);
            uint32_t (&v1)[16] = *reinterpret_cast<uint32_t(*)[16]>(&v[16]);
            convert_chunk<MODE>(w0, s2, nz2, args.zeros != nullptr, has_s, args.wbias, v0);
            convert_chunk<MODE>(w1, s2, nz2, args.zeros != nullptr, has_s, args.wbias, v1);
            if (!row_ok) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0;
            }
            tmem_st32(tcol + qq * 32, v);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // empty first: once the MMA thread sees tfull, this group's share
          // of the stage's release has been counted
          mbar_arrive(&sm.empty[s]);
          if constexpr (PAIR) mbar_arrive_remote(tfull_c + ts * 8);
          else mbar_arrive(&sm.tfull[ts]);
        }
        return true;
      };
      // drain the accumulator at the end of an exact chunk or of the unit
      // (every converter warp); false when a wait gave up
      auto drain = [&](bool final_ev) -> bool {
          // ------------------------------------------------ drain an event
          const bool split = final_ev && u.nslots > 1;
          const size_t slot_elems = static_cast<size_t>(NT) * kTileN * BM;
          const uint32_t* part = reinterpret_cast<const uint32_t*>(args.partials);
          // Split tile: each warp takes its place in the arrival order of the
          // tile's contributors for its sub-tile (low half of the counter).
          // The last to arrive adds the others' partial sums to its own
          // accumulator; the others write theirs and then count themselves as
          // written (high half), which the last one waits for.
          int* ctr = args.counters + (static_cast<size_t>(u.tile) * NCTA + rank) * kConvWarps + cw;
          bool reducer = false;
          if (split) {
            int prev_count = 0;
            if (lane == 0) prev_count = atomicAdd(ctr, 1);
            prev_count = __shfl_sync(0xffffffffu, prev_count, 0);
            reducer = (prev_count & 0xffff) == u.nslots - 1;
          }
          // position of this unit among the tile's contributors (K order), and
          // the slot of contributor sl held by lane sl (<= 32 contributors)
          // (a pair's two CTAs keep separate slots: pair slot * NCTA + rank)
          const int my_sl = p.decomp == kSplitK ? u.split : static_cast<int>(wk.me) - u.cfirst;
          const size_t lane_slot =
              reducer && lane < u.nslots ? (slot_index(p, wk, u, lane) * NCTA + rank) * slot_elems : 0;
          // Pull what this drain will read toward L2 while the last MMAs run:
          // the other contributors' partial sums (reducer) and the int32
          // running sum of the earlier chunks (W4A8 with the global copy).
          uint32_t* gi_base = reinterpret_cast<uint32_t*>(args.icopy) +
                              static_cast<size_t>(blockIdx.x) * NT * BM * kTileN;
          for (int bb = grp; bb < NT * nblk; bb += kConvGroups) {
            const int t = LEAN ? 0 : bb / nblk, cc = (bb - t * nblk) * 8;
            const size_t goff = static_cast<size_t>(bb) * 1024 + q * 256 + lane * 4;
            const size_t coff = LEAN ? goff : static_cast<size_t>(t * BM + cc) * kTileN + r * 8;
            if (MODE == kW4A8 && p.gicopy && !first_chunk) {
              prefetch_l2(gi_base + goff);
              prefetch_l2(gi_base + goff + 128);
            }
            if (reducer) {
              for (int sl = 0; sl < u.nslots; ++sl) {
                if (sl == my_sl) continue;
                const size_t sbase =
                    u.nslots <= 32
                        ? static_cast<size_t>(__shfl_sync(
                              0xffffffffu, static_cast<unsigned long long>(lane_slot), sl))
                        : (slot_index(p, wk, u, sl) * NCTA + rank) * slot_elems;
                prefetch_l2(part + sbase + coff);
                if (LEAN) prefetch_l2(part + sbase + coff + 128);
              }
            }
          }
          if (!__all_sync(0xffffffffu, mbar_wait<true>(sm.dfull, ev & 1, abort, args.status))) {
            return false;
          }
          ++ev;
          tc_fence_after();
          if (reducer) {
            // every other contributor has written its partial sums
            bool done = true;
            if (lane == 0) done = wait_count_hi(ctr, u.nslots - 1, abort, args.status);
            if (!__all_sync(0xffffffffu, __shfl_sync(0xffffffffu, done, 0))) {
              return false;
            }
            __threadfence();
          }
          const size_t my_slot =
              split && !reducer ? (own_slot(p, wk, u) * NCTA + rank) * slot_elems : 0;
          // Blocks of 8 accumulator columns over all weight tiles, round-robin
          // over the converter groups.  Global layout of the int32 running
          // sum (and of the partial sums, LEAN): block bb = (t, cc) is 1024
          // words, the 32 rows of lane quadrant q at q * 256, columns 0-3 of
          // each row (16 bytes per lane) first and columns 4-7 128 words
          // further on, so that each 16-byte access of a warp covers 512
          // contiguous bytes; partial sums otherwise: row r of the block
          // holds its 8 columns contiguously at r * 8.
          for (int bb = grp; bb < NT * nblk; bb += kConvGroups) {
            const int t = LEAN ? 0 : bb / nblk, cc = (bb - t * nblk) * 8;
            const uint32_t dcol = tmem + lane_base + t * BM + cc;
            const int64_t nrow = n0 + t * kTileN + r;  // output column
            const size_t goff = static_cast<size_t>(bb) * 1024 + q * 256 + lane * 4;
            const size_t coff = LEAN ? goff : static_cast<size_t>(t * BM + cc) * kTileN + r * 8;
            uint32_t d[8];
            tmem_ld8(dcol, d);
            if (MODE == kW4A8) {
              // add the int32 running sum of the earlier chunks of this unit:
              // in tensor memory, or in this CTA's global scratch
              const uint32_t icol = tmem + lane_base + p.icol + t * BM + cc;
              uint32_t prev[8];
              if (!first_chunk) {
                if (p.gicopy) ld_cg_halves(gi_base + goff, 128, prev);
                else tmem_ld8(icol, prev);
              }
              tmem_wait_ld();
              add_chunk_sums(d, prev, first_chunk);
              if (!final_ev) {
                if (p.gicopy) {
                  st_halves(gi_base + goff, 128, d);
                } else {
                  tmem_st8(icol, d);
                  tmem_wait_st();
                }
                continue;
              }
            } else {
              tmem_wait_ld();
            }
            // d: this unit's sums of the block (int32 or fp32 bits)
            if (split && !reducer) {
              if (LEAN) st_halves(static_cast<uint32_t*>(args.partials) + my_slot + coff, 128, d);
              else st_v8(static_cast<uint32_t*>(args.partials) + my_slot + coff, d);
              continue;
            }
            if (reducer) {
              // add the contributors in K order, this unit's own sums at its place
              uint32_t acc[8];
              for (int sl = 0; sl < u.nslots; ++sl) {
                uint32_t x[8];
                if (sl == my_sl) {
  #pragma unroll
                  for (int i = 0; i < 8; ++i) x[i] = d[i];
                } else {
                  const size_t sbase =
                      u.nslots <= 32
                          ? static_cast<size_t>(__shfl_sync(
                                0xffffffffu, static_cast<unsigned long long>(lane_slot), sl))
                          : (slot_index(p, wk, u, sl) * NCTA + rank) * slot_elems;
                  if (LEAN) ld_cg_halves(part + sbase + coff, 128, x);
                  else ld_cg_v8(part + sbase + coff, x);
                }
  #pragma unroll
                for (int i = 0; i < 8; ++i) {
                  if (sl == 0) acc[i] = x[i];
                  else if (MODE == kW4A8)
                    acc[i] = static_cast<uint32_t>(static_cast<int32_t>(acc[i]) +
                                                   static_cast<int32_t>(x[i]));
                  else
                    acc[i] = __float_as_uint(__uint_as_float(acc[i]) + __uint_as_float(x[i]));
                }
              }
  #pragma unroll
              for (int i = 0; i < 8; ++i) d[i] = acc[i];
            }
            // outputs
  #pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int64_t m = m0 + cc + i;
              if (nrow < N && m < M)
                store_out<MODE>(args, m, nrow, __uint_as_float(d[i]), static_cast<int32_t>(d[i]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (PAIR) mbar_arrive_remote(dempty_c);
            else mbar_arrive(sm.dempty);
          }
          first_chunk = false;
          if (split && !reducer) {
            // partial sums visible device-wide, then counted as written
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicAdd(ctr, 0x10000);
          } else if (reducer) {
            if (lane == 0) *ctr = 0;  // leave the counter at zero for the next call
          }
        return true;
      };
      if constexpr (kOwnStages) {
        // Exact chunks (W4A8) or the whole unit, each ended by a drain;
        // within a chunk this group visits only its own stages (every
        // kConvGroups-th one): stepping over the other groups' stages one by
        // one cost about as much as converting its own.
        for (int c0 = 0; ok && c0 < nkb; c0 += chunk_len) {
          const int c1 = c0 + chunk_len < nkb ? c0 + chunk_len : nkb;
          int j = c0 + static_cast<int>((static_cast<uint32_t>(grp) + kConvGroups -
                                         (it_u + c0) % kConvGroups) % kConvGroups);
          uint32_t it = it_u + j;
          // ring positions of stage it (divisions once per chunk, then steps
          // of kConvGroups <= S stages): shared-memory slot it % S and its
          // phase, tensor-memory slot it % TS, and the slot and phase of
          // stage it - TS
          uint32_t cs = it % S, cph = (it / S) & 1u, cts = it % TS, ps = 0, pph = 0;
          if (it >= static_cast<uint32_t>(TS)) {
            ps = (it - TS) % S;
            pph = ((it - TS) / S) & 1u;
          }
          for (; j < c1; j += kConvGroups, it += kConvGroups) {
            if (!conv_stage(j, it, cs, cph, cts, ps, pph)) {
              ok = false;
              break;
            }
            // the next stage of this group, kConvGroups further on
            cs += kConvGroups;
            if (cs >= static_cast<uint32_t>(S)) {
              cs -= S;
              cph ^= 1u;
            }
            cts += kConvGroups;
            while (cts >= static_cast<uint32_t>(TS)) cts -= TS;
            const uint32_t itn = it + kConvGroups;
            if (it >= static_cast<uint32_t>(TS)) {
              ps += kConvGroups;
              if (ps >= static_cast<uint32_t>(S)) {
                ps -= S;
                pph ^= 1u;
              }
            } else if (itn >= static_cast<uint32_t>(TS)) {
              ps = (itn - TS) % S;
              pph = ((itn - TS) / S) & 1u;
            }
          }
          if (!ok) break;
          if (!drain(c1 == nkb)) {
            ok = false;
            break;
          }
        }
      } else {
        // every stage in turn, converting this group's (the single-CTA W4A8
        // kernels: the loop above needs more registers there and spills)
        uint32_t it = it_u;
        uint32_t cs = it % S, cph = (it / S) & 1u, cts = it % TS, ps = 0, pph = 0;
        if (it >= static_cast<uint32_t>(TS)) {
          ps = (it - TS) % S;
          pph = ((it - TS) / S) & 1u;
        }
        int cleft = 0;  // stages left in the current exact chunk
        for (int j = 0; j < nkb; ++j, ++it) {
          if (cleft == 0) cleft = chunk_len < nkb - j ? chunk_len : nkb - j;
          if (static_cast<int>(it % kConvGroups) == grp &&
              !conv_stage(j, it, cs, cph, cts, ps, pph)) {
            ok = false;
            break;
          }
          if (++cs == static_cast<uint32_t>(S)) {
            cs = 0;
            cph ^= 1u;
          }
          if (++cts == static_cast<uint32_t>(TS)) cts = 0;
          if (it + 1 > static_cast<uint32_t>(TS) && ++ps == static_cast<uint32_t>(S)) {
            ps = 0;
            pph ^= 1u;
          }
          if (--cleft != 0) continue;
          if (!drain(j == nkb - 1)) {
            ok = false;
            break;
          }
        }
      }
      it_u += nkb;
    }
  }

  tc_fence_before();
  // a pair: neither CTA frees its tensor memory or exits while the other may
  // still arrive on its barriers or the MMAs may read its shared memory
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  if (warp == kProdWarp) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}


namespace {
template <int MODE, bool MMA2, bool PAIR, bool LEAN = false>
cudaError_t launch_tc_mode(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                           const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s) {
  auto* fn = &tc_gemm_kernel<MODE, MMA2, PAIR, LEAN>;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan.smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (MODE == kW4A8) {
    // W4A8: a programmatic dependent of its int8 -> bf16 staging launch; only
    // the activation producer waits for that grid (weights and scales are not
    // written by it), so the weight stream starts at once
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, fn, amap, smap, zmap, plan, args);
}

// fp8 activations are read by TMA straight from the caller's buffer; W4A8
// int8 from the workspace's bf16 copy; W4A16 from the caller's buffer.
template <bool MMA2, bool PAIR = false>
cudaError_t launch_tc_t(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                        const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s) {
  // CTA pairs: LEAN except for per-channel W4A8 (see tc_gemm_kernel)
  switch (plan.mode) {
    case kW4A16_F16:
      return launch_tc_mode<kW4A16_F16, MMA2, PAIR, PAIR>(plan, amap, smap, zmap, args, s);
    case kW4A16_BF16:
      return launch_tc_mode<kW4A16_BF16, MMA2, PAIR, PAIR>(plan, amap, smap, zmap, args, s);
    case kW4A8F8: return launch_tc_mode<kW4A8F8, MMA2, PAIR, PAIR>(plan, amap, smap, zmap, args, s);
    default:
      if (PAIR && tc_grouped(plan))
        return launch_tc_mode<kW4A8, MMA2, PAIR, PAIR>(plan, amap, smap, zmap, args, s);
      return launch_tc_mode<kW4A8, MMA2, PAIR>(plan, amap, smap, zmap, args, s);
  }
}

// Most two-CTA clusters of the pair kernel of this mode that can be resident
// at once with `smem` bytes of shared memory per CTA (-1 when unknown).
template <int MODE>
int tc_pair_clusters_mode(size_t smem) {
  auto* fn = &tc_gemm_kernel<MODE, false, true>;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return n;
}
}  // namespace

}  // namespace w4
