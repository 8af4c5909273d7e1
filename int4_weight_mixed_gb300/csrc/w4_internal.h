// w4_internal.h — plan and launch interfaces shared by the host library
// (w4_api.cu) and the kernels (w4_kernels.cu, w4_tc.cu).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4 {

constexpr int kLayoutVersion = 1;
// Prepacked tile: 128 weight columns (n) x 32 K-values per 16-byte chunk;
// buffer order [N/128][K/32][128][4 words].  Within each 32-bit word the
// eight K-values k0..k0+7 sit in ExLlama order: value j at bits
// (j/2)*4 + (j%2)*16, so bits 0-3/16-19 hold the pair (k0, k0+1), bits
// 4-7/20-23 the pair (k0+2, k0+3), and so on.
constexpr int kTileN = 128;
constexpr int kChunkK = 32;
constexpr int kStageK = 64;   // K granularity: one 128-byte swizzled activation row
constexpr int kMaxStages = 32;
constexpr int kMaxTmemStages = 8;
// Converter warps work in groups of four (one warp per tensor-memory lane
// quadrant); group g converts the pipeline stages it with
// it % kConvGroups == g, so kConvGroups stages are in conversion at once.
constexpr int kConvGroups = 4;
constexpr int kConvWarps = 4 * kConvGroups;
// warps 0..kConvWarps-1: converters / epilogue (four warpgroups); then the
// weight producer (also allocates tensor memory), the MMA issuer, the
// activation producer and the second MMA-issuing warp (the two issuers
// alternate by MMA group; idle in the one-issuer kernel) — the fifth warpgroup
constexpr int kTcThreads = 32 * kConvWarps + 128;
constexpr int kProdWarp = kConvWarps;
constexpr int kMmaWarp = kConvWarps + 1;
constexpr int kActWarp = kConvWarps + 2;
constexpr int kMma2Warp = kConvWarps + 3;
// Registers a thread after the split at kernel start (setmaxnreg): the
// launch gives every thread 96 (640 threads, five warps on a sub-partition);
// the converter warpgroups take 104, the fifth warpgroup keeps 64:
// 512 * 104 + 128 * 64 = 61440 <= 640 * 96 = 61440.
constexpr int kTcLaunchRegs = 96;
constexpr int kTcConvRegs = 104;
constexpr int kTcOtherRegs = 64;
static_assert(32 * kConvWarps * kTcConvRegs + 128 * kTcOtherRegs <= kTcThreads * kTcLaunchRegs,
              "register split exceeds the launch allocation");
constexpr size_t kWsHeader = 256;                // status word + spare
// Split-K tile counters after the header: zero on entry, left zero by every
// call (and re-zeroed by w4_check_status after a timeout).
constexpr size_t kCounterBytes = 64 * 1024;

enum Mode { kW4A16_F16 = 0, kW4A16_BF16 = 1, kW4A8 = 2, kW4A8F8 = 3 };  // kW4A8F8: E4M3 activations

enum Engine { kEngineSimt = 0, kEngineTc = 1, kEngineDk = 2, kEngineDs = 3, kEngineGv = 4 };
enum Decomp { kDataParallel = 0, kStreamK = 1, kSplitK = 2 };

struct Schedule {
  const char* name;
  int engine;
  int bm;      // activation rows per tile (UMMA N)
  int decomp;  // kDataParallel / kStreamK / kSplitK
  int nt;      // 128-column weight tiles per CTA (tc): 1, or 2 to share each activation tile
  int pair;    // tc: 1 = two CTAs of a cluster share each MMA (tile of 256 weight columns)
};

// Everything a tc launch needs, computed on the host.
struct TcPlan {
  int mode;
  int bm;
  int nt;              // 128-column weight tiles per CTA tile (1 or 2)
  int pair;            // CTA pairs (cta_group::2): tile = 2 x nt x 128 weight columns,
                       // each CTA holding bm / 2 activation rows; grid = 2 x pairs
  int n128;            // ceil(N / 128): prepacked weight tiles that exist
  int ksplit;          // kSplitK: K splits per tile
  int icol;            // W4A8: first tensor-memory column of the int32 copies (0 = none)
  int gicopy;          // W4A8: int32 copies in global scratch instead (tensor memory full)
  int nsub;            // 64-wide K blocks per pipeline stage (1, 2 or 4)
  int stages;          // shared-memory pipeline stages
  int tstages;         // tensor-memory A stages (nsub * 32 columns each)
  int acol;            // first tensor-memory column of the A stages
  int gps;             // scale / zero-point rows per stage (groups it spans)
  int a3d;             // activations as one 3-D box {64, BM, nsub} per stage
  int m_tiles, n_tiles, tiles;
  int kb_total;        // pipeline stages per tile: ceil(K / (64 * nsub))
  int k64;             // K / 64
  int grid;            // CTAs
  int decomp;
  int max_segs;        // partial slots per CTA (stream-K)
  int chunk_stages;    // W4A8: stages per exact fp32 accumulation chunk
  size_t smem_bytes;
  size_t ws_counters;  // byte offsets into the workspace
  size_t ws_partials;
  size_t ws_act;       // W4A8 bf16 activations
  size_t ws_icopy;     // W4A8 int32 running sums (gicopy): grid x NT*BM*128 x 4 bytes
  size_t ws_total;
};

// MMA groups issued by two alternating threads (else one): where a group's
// MMAs are short (N <= 128 activation rows)
inline bool tc_mma2(const TcPlan& p) { return p.bm <= 128 && !p.pair; }
// W4A8 with group scales: exact chunks of 1024 K (16384 K per-channel)
inline bool tc_grouped(const TcPlan& p) { return p.chunk_stages * kStageK * p.nsub < 16384; }

struct TcArgs {
  const uint8_t* b_packed;
  const void* scales;      // W4A16 [G][N] 16-bit; W4A8 int8 sg [G][N] or null
  const void* zeros;       // W4A16 [G][N] 16-bit or null
  const float* s_tok;      // W4A8
  const float* s_ch;       // W4A8
  void* out;
  const void* bias;        // [N] of the output type, added before rounding, or null
  int out_s32;             // W4A8 raw int32 output
  int wbias;               // 8 for uint4b8 / int4 (offset binary), 0 for uint4
  int64_t M, N, K;
  int64_t group_size;
  int* status;
  int* counters;
  void* partials;
  int32_t* icopy;          // tc W4A8 with gicopy: per-CTA int32 running sums
};

// Skinny-M schedule (mma.sync, weights dequantized into register fragments).
struct DkPlan {
  int mode;
  int nj;        // 8-row activation tiles: M <= 8 * nj
  int n_tiles;   // 128-column weight tiles
  int kblocks;   // 128-wide K blocks: ceil(K / 128)
  int ksplit;    // K splits per tile (units = n_tiles * ksplit = grid)
  int kbu_max;   // largest number of K blocks in one unit
  int grid;
  size_t smem_bytes;
};

// Streamed skinny-M schedule (bulk-copied weight stages, mma.sync, stream-K).
// CTAs per SM: three for up to 8 activation rows (about 110 registers a
// thread), two for up to 16 (about 150), one of ten warps for up to 32
__host__ __device__ constexpr int ds_ctas_per_sm(int nj) { return nj == 1 ? 3 : nj == 2 ? 2 : 1; }
__host__ __device__ constexpr size_t ds_smem_budget(int nj) {
  return nj == 1 ? 72 * 1024 : nj == 2 ? 108 * 1024 : 216 * 1024;
}
struct DsPlan {
  int mode;
  int nj;          // 8-row activation tiles: M <= 8 * nj
  int n_tiles;     // 128-column weight tiles
  int kblocks;     // 128-wide K blocks: ceil(K / 128)
  int sb;          // K blocks per pipeline stage
  int stages;      // shared-memory pipeline stages
  int grid;        // persistent CTAs (two per SM)
  int max_segs;    // tiles touched by one CTA (partial slots per CTA)
  size_t smem_bytes;
  size_t ws_partials, ws_prep, ws_total;  // workspace byte offsets / size
};

// Clustered skinny-M schedule (one launch: each 128-column tile split along K
// over a cluster of `cluster` CTAs, reduced through distributed shared
// memory).
// CTAs per SM of the clustered skinny-M kernel: four for up to 8 rows, three
// for up to 16, two for up to 32
__host__ __device__ constexpr int gv_ctas_per_sm(int nj) { return nj == 1 ? 4 : nj == 2 ? 3 : 2; }
struct GvPlan {
  int mode;
  int nj;          // 8-row activation tiles: M <= 8 * nj
  int n_tiles;     // 128-column weight tiles
  int kblocks;     // 128-wide K blocks: ceil(K / 128)
  int cluster;     // CTAs per tile (cluster size, 1..16)
  int stages;      // shared-memory pipeline stages
  int grid;        // n_tiles * cluster
  size_t smem_bytes;
};

// Host launchers (return cudaError_t of the launch).
cudaError_t launch_prepack(const int32_t* w_q, int wtype, int layout, int64_t K, int64_t N,
                           uint8_t* out, cudaStream_t s);
cudaError_t launch_unprepack(const uint8_t* packed, int wtype, int layout, int64_t K,
                             int64_t N, int32_t* w_q, cudaStream_t s);
cudaError_t launch_simt(int mode, const void* a, const TcArgs& args, cudaStream_t s);
// K == 0 with a bias: out[m][n] = bias[n] (W4A16), fp16_rn(0 * s_tok * s_ch + bias) (W4A8)
cudaError_t launch_bias_rows(int mode, int64_t M, int64_t N, const void* bias, bool w4a8,
                             void* out, cudaStream_t s);
cudaError_t launch_a8_to_bf16(const int8_t* a, int64_t count, void* out, cudaStream_t s);
// out: 0 int8 codes, 1 int8 codes as bf16 values, 2 E4M3 codes
cudaError_t launch_quant_per_token(bool bf16, const void* a, int64_t M, int64_t K, void* q,
                                   float* s_tok, int out, cudaStream_t s);
cudaError_t launch_tc(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                      const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s);
cudaError_t launch_dk(const DkPlan& plan, const void* a, const TcArgs& args, cudaStream_t s);
size_t dk_smem_bytes(int nj, int kbu_max);
cudaError_t launch_ds(const DsPlan& plan, const void* a, const TcArgs& args, uint8_t* prep,
                      cudaStream_t s);
size_t ds_smem_bytes(int sb, int nj, int m, int stages);
size_t ds_prep_bytes(int nj, int m, int kblocks);
size_t gv_smem_bytes(int nj, int mode, int stages);
int gv_max_clusters(int mode, int nj, int C, size_t smem);
cudaError_t launch_gv(const GvPlan& plan, const CUtensorMap& amap, const TcArgs& args,
                      cudaStream_t s);
size_t tc_stage_bytes(int bm, int nsub, int nt, int wblk);
size_t tc_smem_bytes(int bm, int nsub, int nt, int stages, int wblk);
int tc_max_stages(int bm, int nsub, int nt, int wblk);
// Most co-resident two-CTA clusters of the pair kernel (-1 without a device).
int tc_pair_clusters(int mode, size_t smem);

}  // namespace w4
