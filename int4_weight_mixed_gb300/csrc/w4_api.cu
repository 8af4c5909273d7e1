// w4_api.cu — the C ABI of libw4 (declared in include/w4.h): argument
// validation, the schedule table and default heuristic, workspace planning,
// tensor-map creation and kernel launch.  No allocation happens here: the
// caller owns every buffer.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <string>

#include "../../include/w4.h"
#include "w4_internal.h"

namespace w4 {
namespace {

thread_local std::string g_last_error;

w4_status fail(w4_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

w4_status cuda_fail(cudaError_t e, const char* what) {
  return fail(W4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Schedules ("Machete Readme", "Code Generation": a set of schedule configs
// with a default heuristic and an optional explicit choice).
const Schedule kSchedules[] = {
    {"simt", kEngineSimt, 0, kDataParallel, 1},       {"tc16_sk", kEngineTc, 16, kStreamK, 1},
    {"tc32_sk", kEngineTc, 32, kStreamK, 1},          {"tc64_sk", kEngineTc, 64, kStreamK, 1},
    {"tc128_sk", kEngineTc, 128, kStreamK, 1},        {"tc128_dp", kEngineTc, 128, kDataParallel, 1},
    {"tc256_sk", kEngineTc, 256, kStreamK, 1},        {"tc256_dp", kEngineTc, 256, kDataParallel, 1},
    {"dk8_sk", kEngineDk, 8, kStreamK, 1},            {"dk16_sk", kEngineDk, 16, kStreamK, 1},
    {"tc128x2_sk", kEngineTc, 128, kStreamK, 2},      {"tc128x2_dp", kEngineTc, 128, kDataParallel, 2},
    {"tc128x2_kp", kEngineTc, 128, kSplitK, 2},
    {"ds8_sk", kEngineDs, 8, kStreamK, 1},            {"ds16_sk", kEngineDs, 16, kStreamK, 1},
    {"tc256_kp", kEngineTc, 256, kSplitK, 1},
    {"ds32_sk", kEngineDs, 32, kStreamK, 1},
    {"gv8_cl", kEngineGv, 8, kSplitK, 1},             {"gv16_cl", kEngineGv, 16, kSplitK, 1},
    {"gv32_cl", kEngineGv, 32, kSplitK, 1},
    // two CTAs of a cluster share each MMA (cta_group::2): 256 weight columns
    // x 256 activation rows per tile, 128 activation rows per CTA
    {"tc256p_sk", kEngineTc, 256, kStreamK, 1, 1},    {"tc256p_dp", kEngineTc, 256, kDataParallel, 1, 1},
    // the same with 128 activation rows (64 per CTA): the accumulator is half
    // as wide, so the W4A8 int32 running sum stays in tensor memory beside it
    {"tc128p_sk", kEngineTc, 128, kStreamK, 1, 1},
};
constexpr int kNumSchedules = sizeof(kSchedules) / sizeof(kSchedules[0]);

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;  // GB300
  }
  return n;
}

int mode_of(int a_type) {
  return a_type == W4_F16    ? kW4A16_F16
         : a_type == W4_BF16 ? kW4A16_BF16
         : a_type == W4_E4M3 ? kW4A8F8
                             : kW4A8;
}
bool valid_a_type(int a_type) {
  return a_type == W4_F16 || a_type == W4_BF16 || a_type == W4_S8 || a_type == W4_E4M3;
}

TcPlan make_plan(int si, int mode, int64_t M, int64_t N, int64_t K, int64_t gs);
DkPlan make_dk_plan(int si, int mode, int64_t M, int64_t N, int64_t K, size_t* ws_partials,
                    size_t* ws_total);
constexpr size_t kMaxDynSmem = 227 * 1024;  // dynamic shared memory a CTA may opt into

// Whether schedule `si` can run this (already validated) problem shape.
bool schedule_fits(int si, int mode, int64_t M, int64_t N, int64_t K, int64_t gs, bool has_sg) {
  const Schedule& sc = kSchedules[si];
  if (sc.engine == kEngineSimt) return true;
  // fp8 activations: the clustered skinny-M and the tensor-core schedules
  if (mode == kW4A8F8 && sc.engine != kEngineGv && sc.engine != kEngineTc) return false;
  if (sc.engine == kEngineDk) {  // M rows in 8-row tiles; a 128-wide K block in one group
    if (M > sc.bm || (gs != K && gs % 128 != 0)) return false;
    size_t wp, wt;  // and the staged activations of a unit fit in shared memory
    return make_dk_plan(si, mode, M, N, K, &wp, &wt).smem_bytes <= kMaxDynSmem;
  }
  if (sc.engine == kEngineDs || sc.engine == kEngineGv)  // also bulk copies of 16-byte-multiple scale rows
    return M <= sc.bm && (gs == K || gs % 128 == 0) && N % 8 == 0 &&
           !(mode == kW4A8 && has_sg && N % 16 != 0);
  if (N % 8 != 0) return false;                      // 16-byte scale rows
  if (mode == kW4A8 && has_sg && N % 16 != 0) return false;
  // tensor memory must hold the accumulators (and the W4A8 int32 copies)
  // beside at least one stage of converted weights
  return make_plan(si, mode, M, N, K, gs).tstages >= 1;
}

// Build the launch plan of a tc schedule.
TcPlan make_plan_uncached(int si, int mode, int64_t M, int64_t N, int64_t K, int64_t gs) {
  const Schedule& sc = kSchedules[si];
  TcPlan p{};
  p.mode = mode;
  p.bm = sc.bm;
  p.nt = sc.nt;
  p.pair = sc.pair;
  const int ncta = p.pair ? 2 : 1;
  const int bmc = p.bm / ncta;  // activation rows in each CTA's shared memory
  // K block: 64 16-bit values (4 KB of nibbles per tile), or 128 E4M3 values
  // (8 KB) for fp8 activations
  const int bk = mode == kW4A8F8 ? 128 : kStageK;
  const int wblk = mode == kW4A8F8 ? 8192 : 4096;
  // K depth of a pipeline stage: skinny tiles need >= 8 KB of nibbles per
  // stage to hide the per-stage cost of the producer; wide tiles are
  // compute-bound and take shallower stages so that several fit in shared
  // memory.
  int nsub = p.bm <= 64 ? 4 : (p.bm <= 128 ? 2 : 1);
  nsub = nsub / p.nt > 0 ? nsub / p.nt : 1;
  const int64_t G = K / gs;
  auto group_ok = [&](int ns) {  // a stage covers whole groups or lies inside one
    return G <= 1 || (ns * kStageK) % gs == 0 || gs % (ns * kStageK) == 0;
  };
  while (nsub > 1 && !group_ok(nsub)) nsub /= 2;
  // The converter groups need at least kConvGroups stages in shared memory
  // (the order of their barrier waits relies on it): shallower stages when
  // the deep ones do not fit that many times.
  while (nsub > 1 && tc_max_stages(bmc, nsub, p.nt, wblk) < kConvGroups) {
    nsub /= 2;
    while (nsub > 1 && !group_ok(nsub)) nsub /= 2;
  }
  p.nsub = nsub;
  p.gps = (G > 1 && gs < nsub * kStageK) ? static_cast<int>(nsub * kStageK / gs) : 1;
  p.stages = tc_max_stages(bmc, nsub, p.nt, wblk);
  p.smem_bytes = tc_smem_bytes(bmc, nsub, p.nt, p.stages, wblk);
  p.m_tiles = static_cast<int>((M + p.bm - 1) / p.bm);
  p.n128 = static_cast<int>((N + kTileN - 1) / kTileN);
  p.n_tiles = (p.n128 + p.nt * ncta - 1) / (p.nt * ncta);
  p.tiles = p.m_tiles * p.n_tiles;
  p.k64 = static_cast<int>(K / bk);
  p.kb_total = (p.k64 + nsub - 1) / nsub;
  // W4A8 exactness: |a| <= 128 and |v*sg| <= 128 (group) or |v| <= 8
  // (per-channel) keep every fp32 partial sum of a chunk within 2^24.
  p.chunk_stages = static_cast<int>(((gs < K) ? 1024 : 16384) / (kStageK * nsub));
  // units of work distribution: CTAs, or the two-CTA clusters that can be
  // resident at once
  int sms = sm_count();
  if (p.pair) {
    // queried once per mode (a pair plan's shared memory depends on the mode
    // only); without a device, one pair per two SMs
    static std::mutex mu;
    static int cache[4];  // resident clusters + 1 (0: not yet queried)
    std::lock_guard<std::mutex> lock(mu);
    if (cache[mode] == 0) {
      const int c = tc_pair_clusters(mode, p.smem_bytes);
      cache[mode] = (c > 0 ? c : sms / 2) + 1;
    }
    sms = cache[mode] - 1;
  }
  p.decomp = sc.decomp;
  if (p.tiles * static_cast<size_t>(kConvWarps) * 4 * ncta > kCounterBytes)
    p.decomp = kDataParallel;
  p.ws_counters = kWsHeader;
  p.ws_partials = p.ws_counters + kCounterBytes;
  p.ksplit = 1;
  p.max_segs = 1;
  size_t part = 0;
  const size_t slot_bytes = static_cast<size_t>(p.nt) * kTileN * p.bm * 4;
  if (p.decomp == kDataParallel) {
    p.grid = (p.tiles < sms ? p.tiles : sms) * ncta;
  } else if (p.decomp == kSplitK) {
    // K splits: W4A8 splits at least until no unit is longer than one exact
    // chunk; then the split count minimizes waves x stages per unit, with a
    // charge for writing the partial sums when there is more than one split.
    int ks_min = 1;
    if (mode == kW4A8) ks_min = (p.kb_total + p.chunk_stages - 1) / p.chunk_stages;
    double best = 1e30;
    int best_ks = ks_min;
    for (int ks = ks_min; ks <= 16 && ks <= p.kb_total; ++ks) {
      const int64_t units = static_cast<int64_t>(p.tiles) * ks;
      const int64_t waves = (units + sms - 1) / sms;
      const int kbu = (p.kb_total + ks - 1) / ks;
      // a partial-sum slot costs about as much as a dozen stages to write
      const double cost = static_cast<double>(waves) * (kbu + 8 + (ks > 1 ? 12 : 0));
      if (cost < best) {
        best = cost;
        best_ks = ks;
      }
    }
    p.ksplit = best_ks;
    const int64_t units = static_cast<int64_t>(p.tiles) * p.ksplit;
    p.grid = static_cast<int>(units < sms ? units : sms) * ncta;
    if (p.ksplit > 1) part = static_cast<size_t>(p.tiles) * p.ksplit * slot_bytes * ncta;
  } else {
    const int64_t T = static_cast<int64_t>(p.tiles) * p.kb_total;
    int64_t g = T / 2;  // at least 2 stages per CTA (pair)
    if (g > sms) g = sms;
    if (g < 1) g = 1;
    p.grid = static_cast<int>(g) * ncta;
    int ms = 1;
    for (int64_t c = 0; c < g; ++c) {
      int64_t b = c * T / g, e = (c + 1) * T / g;
      if (e <= b) continue;
      int segs = static_cast<int>((e - 1) / p.kb_total - b / p.kb_total + 1);
      if (segs > ms) ms = segs;
    }
    p.max_segs = ms;
    part = static_cast<size_t>(p.grid) * p.max_segs * slot_bytes;  // one slot set per CTA
  }
  // Tensor memory: accumulators (NT x BM columns), the W4A8 int32 copies
  // when a unit can span several exact chunks, then the converted-weight
  // stages (NT x nsub x 32 columns each).
  bool long_units = p.kb_total > p.chunk_stages;
  if (p.decomp == kSplitK) long_units = (p.kb_total + p.ksplit - 1) / p.ksplit > p.chunk_stages;
  const int dcols = p.nt * p.bm;
  // W4A8 units longer than one exact chunk keep an int32 running sum: in
  // tensor memory beside the accumulators when that leaves two or more
  // converted-weight stages, else in a per-CTA global scratch (its owner
  // thread writes and reads it back, one element per accumulator cell).
  const bool need_i = mode == kW4A8 && long_units;
  const bool tmem_i = need_i && 512 - 2 * dcols >= 2 * p.nt * nsub * 32;
  p.icol = tmem_i ? dcols : 0;
  p.gicopy = need_i && !tmem_i ? 1 : 0;
  const int used = (p.icol ? 2 * dcols : dcols);
  p.acol = (used + 31) / 32 * 32;
  int ts = p.acol >= 512 ? 0 : (512 - p.acol) / (p.nt * nsub * 32);
  if (p.ksplit > 16) ts = 0;  // too many partial sums to be worth it: not offered
  if (ts > kMaxTmemStages) ts = kMaxTmemStages;
  if (ts > p.stages - 1) ts = p.stages - 1;
  if (p.stages < kConvGroups) ts = 0;  // not offered (see above)
  p.tstages = ts;
  p.ws_act = align256(p.ws_partials + part);
  size_t act = mode == kW4A8 ? static_cast<size_t>(M) * K * 2 : 0;
  p.ws_icopy = align256(p.ws_act + act);
  const size_t icopy = p.gicopy ? static_cast<size_t>(p.grid) * dcols * kTileN * 4 : 0;
  p.ws_total = align256(p.ws_icopy + icopy);
  return p;
}

// The plan of a tc schedule, remembered per shape and device: a call plans
// its schedule several times (fit, workspace, launch), each a few
// microseconds of host time.
TcPlan make_plan(int si, int mode, int64_t M, int64_t N, int64_t K, int64_t gs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  const auto key = std::make_tuple(si, mode, M, N, K, gs, dev);
  static std::mutex mu;
  static std::map<decltype(key), TcPlan> cache;
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const TcPlan p = make_plan_uncached(si, mode, M, N, K, gs);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 4096) cache.clear();
  cache.emplace(key, p);
  return p;
}

size_t simt_ws_bytes() { return kWsHeader; }
// Plan of the skinny-M (mma.sync) schedule: 128-column tiles x K splits,
// two CTAs per SM; the split count minimizes waves x blocks per unit with a
// small penalty per split (partials and the reduction).
DkPlan make_dk_plan(int si, int mode, int64_t M, int64_t N, int64_t K, size_t* ws_partials,
                    size_t* ws_total) {
  DkPlan p{};
  p.mode = mode;
  p.nj = kSchedules[si].bm / 8;
  p.n_tiles = static_cast<int>((N + kTileN - 1) / kTileN);
  p.kblocks = static_cast<int>((K + 127) / 128);
  const int slots = 2 * sm_count();
  double best = 1e30;
  int best_s = 1;
  for (int ks = 1; ks <= 64 && ks <= p.kblocks; ++ks) {
    // a K split counts its contributors in one counter per weight tile
    if (ks > 1 && static_cast<size_t>(p.n_tiles) * 4 > kCounterBytes) break;
    const int kbu = (p.kblocks + ks - 1) / ks;
    if (dk_smem_bytes(p.nj, kbu) > 100 * 1024) continue;
    const int64_t units = static_cast<int64_t>(p.n_tiles) * ks;
    const int64_t waves = (units + slots - 1) / slots;
    // a wave costs its K blocks plus a fixed prologue / epilogue (~6 blocks)
    const double cost = static_cast<double>(waves) * (kbu + 6) * (1.0 + 0.01 * ks);
    if (cost < best) {
      best = cost;
      best_s = ks;
    }
  }
  p.ksplit = best_s;
  p.kbu_max = (p.kblocks + p.ksplit - 1) / p.ksplit;
  p.grid = p.n_tiles * p.ksplit;
  p.smem_bytes = dk_smem_bytes(p.nj, p.kbu_max);
  (void)M;
  const size_t part = p.ksplit > 1 ? static_cast<size_t>(p.ksplit) * p.n_tiles * 8 * p.nj *
                                         kTileN * 4
                                   : 0;
  *ws_partials = kWsHeader + kCounterBytes;
  *ws_total = align256(*ws_partials + part);
  return p;
}

// Plan of the streamed skinny-M schedule: two or three persistent CTAs per SM over a
// stream-K split of the (128-column tile, 128-K block) iterations.
DsPlan make_ds_plan(int si, int mode, int64_t M, int64_t N, int64_t K) {
  DsPlan p{};
  p.mode = mode;
  p.nj = kSchedules[si].bm / 8;
  p.n_tiles = static_cast<int>((N + kTileN - 1) / kTileN);
  p.kblocks = static_cast<int>((K + 127) / 128);
  // two K blocks (16 KB of nibbles) per stage: each stage costs its producer
  // thread a fixed few hundred nanoseconds, so stages must not be smaller
  p.sb = 2;  // must match the kernel's stage depth
  p.stages = 16;
  while (p.stages > 2 &&
         ds_smem_bytes(p.sb, p.nj, static_cast<int>(M), p.stages) > ds_smem_budget(p.nj))
    --p.stages;
  p.smem_bytes = ds_smem_bytes(p.sb, p.nj, static_cast<int>(M), p.stages);
  const int64_t T = static_cast<int64_t>(p.n_tiles) * p.kblocks;
  // every CTA streams at least eight blocks (four stages): a CTA has a fixed
  // start-up cost, and a tile split over many CTAs a long reduction
  int64_t g = ds_ctas_per_sm(p.nj) * static_cast<int64_t>(sm_count());
  if (g > (T + 7) / 8) g = (T + 7) / 8;
  if (g < 1) g = 1;
  p.grid = static_cast<int>(g);
  int ms = 1;
  for (int64_t c = 0; c < g; ++c) {
    const int64_t b = c * T / g, e = (c + 1) * T / g;
    if (e <= b) continue;
    const int segs = static_cast<int>((e - 1) / p.kblocks - b / p.kblocks + 1);
    if (segs > ms) ms = segs;
  }
  p.max_segs = ms;
  p.ws_partials = kWsHeader + kCounterBytes;
  const size_t part = static_cast<size_t>(p.grid) * p.max_segs * 8 * p.nj * kTileN * 4;
  p.ws_prep = align256(p.ws_partials + part);
  p.ws_total = align256(p.ws_prep + ds_prep_bytes(p.nj, static_cast<int>(M), p.kblocks));
  return p;
}

// Plan of the clustered skinny-M schedule: the cluster size C (CTAs per
// 128-column tile, each streaming an equal share of the tile's K blocks) is
// the smallest that minimizes the K blocks of the busiest CTA while every
// cluster of the grid is resident at once.
GvPlan make_gv_plan(int si, int mode, int64_t M, int64_t N, int64_t K) {
  GvPlan p{};
  p.mode = mode;
  p.nj = kSchedules[si].bm / 8;
  p.n_tiles = static_cast<int>((N + kTileN - 1) / kTileN);
  p.kblocks = static_cast<int>((K + 127) / 128);
  p.stages = p.nj == 1 ? 4 : 3;
  p.smem_bytes = gv_smem_bytes(p.nj, mode, p.stages);
  // resident clusters per cluster size, from the occupancy calculator when a
  // device is present (cached per mode, row tiles and size), else from the
  // design's CTAs per SM
  static std::mutex mu;
  static int cache[4][3][17];  // resident clusters + 1 (0: not yet queried)
  const int mi = mode, ni = p.nj == 1 ? 0 : p.nj == 2 ? 1 : 2;
  const int per_sm = gv_ctas_per_sm(p.nj);
  const int sms = sm_count();
  int best_c = 1, best_nkb = p.kblocks;
  for (int C = 1; C <= 16 && C <= p.kblocks; ++C) {
    int clusters;
    {
      std::lock_guard<std::mutex> lock(mu);
      if (cache[mi][ni][C] == 0) {
        const int q = gv_max_clusters(mode, p.nj, C, p.smem_bytes);
        cache[mi][ni][C] = (q >= 0 ? q : sms * per_sm / C) + 1;
      }
      clusters = cache[mi][ni][C] - 1;
    }
    if (static_cast<int64_t>(p.n_tiles) > clusters) continue;  // more than one wave
    const int nkb = (p.kblocks + C - 1) / C;
    if (nkb < best_nkb) {
      best_nkb = nkb;
      best_c = C;
    }
  }
  p.cluster = best_c;
  p.grid = p.n_tiles * p.cluster;
  (void)M;
  return p;
}

// Per-shape overrides of the default heuristic ("Machete Readme", "Code
// Generation": a default heuristic with per-shape exceptions; the vLLM
// "rdna_hybrid_w4a16" page keeps a table of them, _GFX1X_PREFILL_OVERRIDES).
// Built-in entries come from A/B timings of the candidate schedules on
// GB300 (graphs of 16 back-to-back launches over rotated weight copies, more
// than 2x L2 between two reads of a copy); entries installed at run time
// (w4_override_schedule) are consulted first.  M in [m_lo, m_hi]; group_size
// as resolved (K for one group per column).
struct Override {
  int mode;
  int64_t m_lo, m_hi, N, K, gs;
  int schedule;
};
const char* const kBuiltinOverrideNames[] = {"tc256p_dp", "tc256p_dp"};
const Override kBuiltinOverrides[] = {
    // W4A16 bf16, Llama-3-70B MLP down projection (N=8192, K=28672), M=4096:
    // tc256p_dp 1252 us, tc256p_sk 1349, tc256_sk 1598
    {kW4A16_BF16, 4096, 8192, 8192, 28672, 128, -1},
    // W4A16 bf16, Llama-3-70B MLP gate/up (N=57344, K=8192), M=4096:
    // tc256p_dp 2585 us, tc256p_sk 2594, tc256_sk 3341
    {kW4A16_BF16, 4096, 8192, 57344, 8192, 128, -1},
};
constexpr int kMaxOverrides = 256;
std::mutex g_ov_mutex;
Override g_overrides[kMaxOverrides];
int g_num_overrides = 0;

int schedule_index(const char* name) {
  for (int i = 0; i < kNumSchedules; ++i)
    if (strcmp(kSchedules[i].name, name) == 0) return i;
  return -1;
}

bool override_matches(const Override& o, int mode, int64_t M, int64_t N, int64_t K, int64_t gs) {
  return o.mode == mode && M >= o.m_lo && M <= o.m_hi && N == o.N && K == o.K && gs == o.gs;
}

// The schedule an override names for this problem, or -1.
int override_for(int mode, int64_t M, int64_t N, int64_t K, int64_t gs) {
  {
    std::lock_guard<std::mutex> lock(g_ov_mutex);
    for (int i = g_num_overrides - 1; i >= 0; --i)  // the latest installed wins
      if (override_matches(g_overrides[i], mode, M, N, K, gs)) return g_overrides[i].schedule;
  }
  for (size_t i = 0; i < sizeof(kBuiltinOverrides) / sizeof(kBuiltinOverrides[0]); ++i)
    if (override_matches(kBuiltinOverrides[i], mode, M, N, K, gs))
      return schedule_index(kBuiltinOverrideNames[i]);
  return -1;
}

int default_schedule_impl(int mode, int64_t M, int64_t N, int64_t K, int64_t gs, bool has_sg) {
  const int ov = override_for(mode, M, N, K, gs);
  if (ov >= 0 && schedule_fits(ov, mode, M, N, K, gs, has_sg)) return ov;
  // skinny M (up to 32 rows with the clustered or streamed schedule, 16 with
  // the register-fed one where neither can run: N not a multiple of 8):
  // warp-level MMAs on dequantized weights
  // The clustered schedule (one launch) wins while its fixed costs dominate:
  // up to 16 rows on at most 16 MiB of packed weights; the streamed one
  // (stream-K with its own reduction launch) keeps more bytes in flight per
  // SM on larger weights.
  const bool small_w = K * N / 2 <= (int64_t{16} << 20);
  for (int eng : {kEngineGv, kEngineDs, kEngineDk})
    for (int si = 1; si < kNumSchedules; ++si)
      if (kSchedules[si].engine == eng &&
          !(eng == kEngineGv && (kSchedules[si].bm > 16 || (!small_w && mode != kW4A8F8))) &&
          schedule_fits(si, mode, M, N, K, gs, has_sg))
        return si;
  int bm = 16;
  while (bm < M && bm < 256) bm *= 2;
  // stream-K balances fewer than four waves of wide tiles; data-parallel beyond
  const int64_t tiles = ((M + bm - 1) / bm) * ((N + kTileN - 1) / kTileN);
  const bool dp = tiles >= 4 * static_cast<int64_t>(sm_count()) && bm >= 128;
  // 256-row tiles on CTA pairs (W4A8 N=8192 K=21760 M=1024: 241 us against
  // 406 for 128-row single-CTA tiles; fp8 M=1024 153 against 221 for
  // single-CTA 256-row tiles; W4A16 prefill 20-23% faster), and 128-row W4A8
  // tiles (M=128: 66.2 against 67.6 us)
  const bool pair = bm == 256 || (bm == 128 && mode == kW4A8);
  for (int pass = 0; pass < 2; ++pass)
    for (int si = 1; si < kNumSchedules; ++si) {
      const Schedule& sc = kSchedules[si];
      if (sc.engine == kEngineTc && sc.bm == bm && (sc.pair != 0) == pair &&
          (pass == 1 || (sc.decomp == kDataParallel) == dp) &&
          schedule_fits(si, mode, M, N, K, gs, has_sg))
        return si;
    }
  for (int si = 1; si < kNumSchedules; ++si)
    if (kSchedules[si].engine == kEngineTc && kSchedules[si].bm == bm &&
        schedule_fits(si, mode, M, N, K, gs, has_sg))
      return si;
  return 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned_to(const void* p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

struct Problem {
  int mode;
  int64_t M, N, K, gs;
  bool has_sg;
};

w4_status validate(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                   int wtype, int64_t N, const void* b_scales, int scale_type,
                   const void* b_zeros, int64_t group_size, const float* s_tok,
                   const float* s_ch, void* out, int out_type, Problem& pr) {
  if (M < 0 || N < 0 || K < 0) return fail(W4_ERR_INVALID_ARGUMENT, "negative size");
  if (!valid_a_type(a_type))
    return fail(W4_ERR_INVALID_ARGUMENT, "a_type must be W4_F16, W4_BF16, W4_S8 or W4_E4M3");
  if (wtype < W4_UINT4B8 || wtype > W4_INT4) return fail(W4_ERR_INVALID_ARGUMENT, "bad wtype");
  if (K % 8 != 0) return fail(W4_ERR_INVALID_ARGUMENT, "K must be a multiple of 8");
  const int64_t gs = (group_size == -1) ? K : group_size;
  if (K > 0 && (gs <= 0 || K % gs != 0))
    return fail(W4_ERR_INVALID_ARGUMENT, "group_size must be -1 or a positive divisor of K");
  pr.mode = mode_of(a_type);
  pr.M = M;
  pr.N = N;
  pr.K = K;
  pr.gs = gs;
  pr.has_sg = b_scales != nullptr;
  if (M == 0 || N == 0) return W4_OK;
  if (!out) return fail(W4_ERR_INVALID_ARGUMENT, "out is null");
  if (pr.mode == kW4A8F8) {
    // W4A8 with E4M3 activations: symmetric weights, one scale per column
    if (wtype == W4_UINT4)
      return fail(W4_ERR_UNSUPPORTED, "W4A8 supports symmetric weights only (int4 / uint4b8)");
    if (b_zeros) return fail(W4_ERR_UNSUPPORTED, "W4A8 takes no zero-points");
    if (b_scales || gs != K)
      return fail(W4_ERR_UNSUPPORTED, "fp8 activations: per-channel weights only");
    if (out_type != W4_F16) return fail(W4_ERR_UNSUPPORTED, "fp8 activations: fp16 output only");
    if (!s_tok || !s_ch)
      return fail(W4_ERR_INVALID_ARGUMENT, "W4A8 fp16 out needs token and channel scales");
    if (K > 0 && (!a || !b_packed))
      return fail(W4_ERR_INVALID_ARGUMENT, "a and b_packed are required");
  } else if (pr.mode != kW4A8) {
    if (out_type != a_type)
      return fail(W4_ERR_INVALID_ARGUMENT, "W4A16: out_type must equal a_type");
    if (K > 0 && (!a || !b_packed || !b_scales))
      return fail(W4_ERR_INVALID_ARGUMENT, "W4A16: a, b_packed and b_scales are required");
    if (scale_type != a_type)
      return fail(W4_ERR_INVALID_ARGUMENT, "W4A16: scale_type must equal a_type");
    if (s_tok || s_ch)
      return fail(W4_ERR_INVALID_ARGUMENT, "W4A16 takes no token or channel scales");
  } else {
    if (wtype == W4_UINT4)
      return fail(W4_ERR_UNSUPPORTED, "W4A8 supports symmetric weights only (int4 / uint4b8)");
    if (b_zeros) return fail(W4_ERR_UNSUPPORTED, "W4A8 takes no zero-points");
    if (out_type == W4_F16) {
      if (!s_tok || !s_ch)
        return fail(W4_ERR_INVALID_ARGUMENT, "W4A8 fp16 out needs token and channel scales");
    } else if (out_type == W4_S32) {
      if (s_tok || s_ch)
        return fail(W4_ERR_INVALID_ARGUMENT, "W4A8 int32 out takes no float scales");
    } else {
      return fail(W4_ERR_UNSUPPORTED, "W4A8 output must be W4_F16 or W4_S32");
    }
    if (b_scales && scale_type != W4_S8)
      return fail(W4_ERR_INVALID_ARGUMENT, "W4A8 group scales must be int8 (W4_S8)");
    if (!b_scales && gs != K)
      return fail(W4_ERR_INVALID_ARGUMENT, "W4A8 per-group needs int8 group scales");
    if (K > 0 && (!a || !b_packed))
      return fail(W4_ERR_INVALID_ARGUMENT, "a and b_packed are required");
  }
  // every kernel reads or writes each array at least element by element;
  // the prepacked weights as 32-bit words
  const uintptr_t asz = (a_type == W4_S8 || a_type == W4_E4M3) ? 1 : 2;
  const uintptr_t osz = (pr.mode == kW4A8 && out_type == W4_S32) ? 4 : 2;
  const uintptr_t ssz = pr.mode == kW4A8 ? 1 : 2;
  if (!aligned_to(a, asz) || !aligned_to(out, osz) || !aligned_to(b_packed, 4) ||
      !aligned_to(b_scales, ssz) || !aligned_to(b_zeros, 2) || !aligned_to(s_tok, 4) ||
      !aligned_to(s_ch, 4))
    return fail(W4_ERR_INVALID_ARGUMENT,
                "a pointer is not aligned to its element size (b_packed: 4 bytes)");
  if (K % kStageK != 0) return fail(W4_ERR_UNSUPPORTED, "K must be a multiple of 64");
  if (pr.mode == kW4A8F8 && K % 128 != 0)
    return fail(W4_ERR_UNSUPPORTED, "fp8 activations: K must be a multiple of 128");
  if (K > 0 && gs % kStageK != 0)
    return fail(W4_ERR_UNSUPPORTED, "group_size must be a multiple of 64 (or K)");
  return W4_OK;
}

size_t ws_needed(int si, const Problem& pr) {
  if (kSchedules[si].engine == kEngineSimt) return simt_ws_bytes();
  if (kSchedules[si].engine == kEngineDk) {
    size_t wp, wt;
    make_dk_plan(si, pr.mode, pr.M, pr.N, pr.K, &wp, &wt);
    return wt;
  }
  if (kSchedules[si].engine == kEngineDs) return make_ds_plan(si, pr.mode, pr.M, pr.N, pr.K).ws_total;
  if (kSchedules[si].engine == kEngineGv) return kWsHeader;  // the status word only
  return make_plan(si, pr.mode, pr.M, pr.N, pr.K, pr.gs).ws_total;
}

}  // namespace
}  // namespace w4

using namespace w4;

extern "C" {

int w4_layout_version(void) { return kLayoutVersion; }

size_t w4_prepacked_size(int64_t K, int64_t N) {
  if (K <= 0 || N <= 0 || K % kStageK != 0) return 0;
  return static_cast<size_t>((N + kTileN - 1) / kTileN * kTileN) * static_cast<size_t>(K / 2);
}

w4_status w4_prepack_B(const int32_t* w_q, int wtype, int in_layout, int64_t K, int64_t N,
                       void* b_packed, void* stream) {
  if (!w_q || !b_packed) return fail(W4_ERR_INVALID_ARGUMENT, "null pointer");
  if (wtype < W4_UINT4B8 || wtype > W4_INT4) return fail(W4_ERR_INVALID_ARGUMENT, "bad wtype");
  if (in_layout < W4_LAYOUT_KN_SEQ || in_layout > W4_LAYOUT_NK_EXLLAMA)
    return fail(W4_ERR_INVALID_ARGUMENT, "bad layout");
  if (K <= 0 || N <= 0 || K % 8 != 0)
    return fail(W4_ERR_INVALID_ARGUMENT, "K and N must be positive, K a multiple of 8");
  if (K % kStageK != 0) return fail(W4_ERR_UNSUPPORTED, "K must be a multiple of 64");
  if (!aligned_to(w_q, 4) || !aligned_to(b_packed, 4))
    return fail(W4_ERR_INVALID_ARGUMENT, "w_q and b_packed must be 4-byte aligned");
  cudaError_t e = launch_prepack(w_q, wtype, in_layout, K, N, static_cast<uint8_t*>(b_packed),
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4_OK : cuda_fail(e, "prepack launch");
}

w4_status w4_unprepack_B(const void* b_packed, int wtype, int out_layout, int64_t K, int64_t N,
                         int32_t* w_q, void* stream) {
  if (!w_q || !b_packed) return fail(W4_ERR_INVALID_ARGUMENT, "null pointer");
  if (wtype < W4_UINT4B8 || wtype > W4_INT4) return fail(W4_ERR_INVALID_ARGUMENT, "bad wtype");
  if (out_layout < W4_LAYOUT_KN_SEQ || out_layout > W4_LAYOUT_NK_EXLLAMA)
    return fail(W4_ERR_INVALID_ARGUMENT, "bad layout");
  if (K <= 0 || N <= 0 || K % 8 != 0)
    return fail(W4_ERR_INVALID_ARGUMENT, "K and N must be positive, K a multiple of 8");
  if (K % kStageK != 0) return fail(W4_ERR_UNSUPPORTED, "K must be a multiple of 64");
  if (!aligned_to(w_q, 4) || !aligned_to(b_packed, 4))
    return fail(W4_ERR_INVALID_ARGUMENT, "w_q and b_packed must be 4-byte aligned");
  cudaError_t e = launch_unprepack(static_cast<const uint8_t*>(b_packed), wtype, out_layout, K,
                                   N, w_q, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4_OK : cuda_fail(e, "unprepack launch");
}

int w4_num_schedules(void) { return kNumSchedules; }

const char* w4_schedule_name(int schedule) {
  if (schedule < 0 || schedule >= kNumSchedules) return nullptr;
  return kSchedules[schedule].name;
}

int w4_default_schedule(int64_t M, int64_t N, int64_t K, int a_type, int64_t group_size) {
  if (M <= 0 || N <= 0 || K <= 0 || K % kStageK != 0) return -1;
  if (!valid_a_type(a_type)) return -1;
  if (a_type == W4_E4M3 && K % 128 != 0) return -1;
  const int64_t gs = group_size == -1 ? K : group_size;
  return default_schedule_impl(mode_of(a_type), M, N, K, gs, gs != K);
}

w4_status w4_override_schedule(int a_type, int64_t m_lo, int64_t m_hi, int64_t N, int64_t K,
                               int64_t group_size, int schedule) {
  if (!valid_a_type(a_type))
    return fail(W4_ERR_INVALID_ARGUMENT, "a_type must be W4_F16, W4_BF16, W4_S8 or W4_E4M3");
  if (m_lo < 1 || m_hi < m_lo || N < 1 || K < 1 || K % kStageK != 0)
    return fail(W4_ERR_INVALID_ARGUMENT, "bad M range or shape");
  const int64_t gs = group_size == -1 ? K : group_size;
  if (gs <= 0 || K % gs != 0) return fail(W4_ERR_INVALID_ARGUMENT, "bad group_size");
  if (schedule >= kNumSchedules)
    return fail(W4_ERR_INVALID_ARGUMENT, "bad schedule index");
  const int mode = mode_of(a_type);
  std::lock_guard<std::mutex> lock(g_ov_mutex);
  // drop earlier entries for exactly this range, then add (schedule >= 0)
  int n = 0;
  for (int i = 0; i < g_num_overrides; ++i) {
    const Override& o = g_overrides[i];
    if (!(o.mode == mode && o.m_lo == m_lo && o.m_hi == m_hi && o.N == N && o.K == K && o.gs == gs))
      g_overrides[n++] = o;
  }
  g_num_overrides = n;
  if (schedule < 0) return W4_OK;
  if (g_num_overrides == kMaxOverrides) return fail(W4_ERR_UNSUPPORTED, "override table full");
  g_overrides[g_num_overrides++] = Override{mode, m_lo, m_hi, N, K, gs, schedule};
  return W4_OK;
}

size_t w4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int a_type, int64_t group_size) {
  Problem pr{};
  pr.mode = mode_of(a_type);
  pr.M = M < 0 ? 0 : M;
  pr.N = N < 0 ? 0 : N;
  pr.K = K < 0 ? 0 : K;
  pr.gs = group_size == -1 ? pr.K : group_size;
  pr.has_sg = pr.gs != pr.K;
  size_t need = kWsHeader;
  if (pr.M == 0 || pr.N == 0 || pr.K == 0 || pr.K % kStageK != 0) return need;
  // Remembered per shape and device (planning every schedule costs tens of
  // microseconds of host time, and callers ask once per call).
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  const auto key = std::make_tuple(pr.M, pr.N, pr.K, pr.gs, pr.mode, dev);
  static std::mutex mu;
  static std::map<decltype(key), size_t> cache;
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  for (int si = 0; si < kNumSchedules; ++si) {
    if (!schedule_fits(si, pr.mode, pr.M, pr.N, pr.K, pr.gs, pr.has_sg)) continue;
    size_t b = ws_needed(si, pr);
    if (b > need) need = b;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 4096) cache.clear();
  cache.emplace(key, need);
  return need;
}

}  // extern "C"

namespace {
// prestaged: W4A8 on the tensor-core schedule with its bf16 activation copy
// already in the workspace (the dynamic-quantization entry point writes it)
w4_status gemm_impl(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                    int wtype, int64_t N, const void* b_scales, int scale_type,
                    const void* b_zeros, int64_t group_size, const float* a_token_scales,
                    const float* ch_scales, const void* bias, void* out, int out_type,
                    void* workspace, size_t workspace_bytes, void* stream, int schedule,
                    bool prestaged = false) {
  Problem pr{};
  w4_status st = validate(a, a_type, M, K, b_packed, wtype, N, b_scales, scale_type, b_zeros,
                          group_size, a_token_scales, ch_scales, out, out_type, pr);
  if (st != W4_OK) return st;
  if (bias) {
    if (pr.mode == kW4A8 && out_type == W4_S32)
      return fail(W4_ERR_INVALID_ARGUMENT, "the raw int32 output takes no bias");
    if (!aligned_to(bias, 2))
      return fail(W4_ERR_INVALID_ARGUMENT, "bias is not aligned to its element size");
  }
  if (schedule >= kNumSchedules) return fail(W4_ERR_INVALID_ARGUMENT, "bad schedule index");
  if (M == 0 || N == 0) return W4_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0 && !bias) {
    const size_t esz = (pr.mode == kW4A8 && out_type == W4_S32) ? 4 : 2;
    cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(M) * N * esz, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "memset");
  }
  if (K == 0) {  // every output is its column's bias
    cudaError_t e = launch_bias_rows(pr.mode, M, N, bias, a_token_scales != nullptr, out, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "bias launch");
  }
  int si = schedule;
  const bool forced = schedule >= 0;
  if (!forced) si = default_schedule_impl(pr.mode, M, N, K, pr.gs, pr.has_sg);
  if (!schedule_fits(si, pr.mode, M, N, K, pr.gs, pr.has_sg))
    return fail(W4_ERR_UNSUPPORTED, "schedule %s cannot run this shape", kSchedules[si].name);
  const bool ptrs_ok = aligned16(a) && aligned16(b_packed) && aligned16(b_scales) &&
                       aligned16(b_zeros);
  if (kSchedules[si].engine != kEngineSimt && !ptrs_ok) {
    if (forced)
      return fail(W4_ERR_UNSUPPORTED, "tensor-core schedules need 16-byte aligned inputs");
    si = 0;
  }
  if (!workspace) return fail(W4_ERR_WORKSPACE, "workspace is null");
  if (!aligned16(workspace)) return fail(W4_ERR_WORKSPACE, "workspace is not 16-byte aligned");
  const size_t need = ws_needed(si, pr);
  if (workspace_bytes < need)
    return fail(W4_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", workspace_bytes, need);

  TcArgs args{};
  args.b_packed = static_cast<const uint8_t*>(b_packed);
  args.scales = b_scales;
  args.zeros = b_zeros;
  args.s_tok = a_token_scales;
  args.s_ch = ch_scales;
  args.out = out;
  args.bias = bias;
  args.out_s32 = (pr.mode == kW4A8 && out_type == W4_S32) ? 1 : 0;
  args.wbias = (wtype == W4_UINT4) ? 0 : 8;
  args.M = M;
  args.N = N;
  args.K = K;
  args.group_size = pr.gs;
  args.status = static_cast<int*>(workspace);
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  if (kSchedules[si].engine == kEngineSimt) {
    cudaError_t e = launch_simt(pr.mode, a, args, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "simt launch");
  }
  if (kSchedules[si].engine == kEngineDk) {
    size_t wp, wt;
    DkPlan dp = make_dk_plan(si, pr.mode, M, N, K, &wp, &wt);
    args.counters = reinterpret_cast<int*>(ws + kWsHeader);
    args.partials = ws + wp;
    static const bool debug = getenv("W4_DEBUG") != nullptr;
    if (debug)
      fprintf(stderr, "w4: %s M=%lld N=%lld K=%lld nj=%d tiles=%d kblocks=%d ksplit=%d grid=%d smem=%zu\n",
              kSchedules[si].name, (long long)M, (long long)N, (long long)K, dp.nj, dp.n_tiles,
              dp.kblocks, dp.ksplit, dp.grid, dp.smem_bytes);
    cudaError_t e = launch_dk(dp, a, args, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "dk launch");
  }
  if (kSchedules[si].engine == kEngineDs) {
    DsPlan dp = make_ds_plan(si, pr.mode, M, N, K);
    args.counters = reinterpret_cast<int*>(ws + kWsHeader);
    args.partials = ws + dp.ws_partials;
    static const bool debug = getenv("W4_DEBUG") != nullptr;
    if (debug)
      fprintf(stderr,
              "w4: %s M=%lld N=%lld K=%lld nj=%d tiles=%d kblocks=%d sb=%d stages=%d grid=%d "
              "segs=%d smem=%zu\n",
              kSchedules[si].name, (long long)M, (long long)N, (long long)K, dp.nj, dp.n_tiles,
              dp.kblocks, dp.sb, dp.stages, dp.grid, dp.max_segs, dp.smem_bytes);
    cudaError_t e = launch_ds(dp, a, args, ws + dp.ws_prep, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "ds launch");
  }

  if (kSchedules[si].engine == kEngineGv) {
    GvPlan gp = make_gv_plan(si, pr.mode, M, N, K);
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return fail(W4_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    CUtensorMap amap;
    CUresult r;
    const cuuint32_t rows = static_cast<cuuint32_t>(8 * gp.nj);
    if (pr.mode == kW4A8 || pr.mode == kW4A8F8) {
      // int8 / E4M3 [M][K]: one box of 128 K x all rows per K block
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
      const cuuint32_t box[2] = {128, rows};
      const cuuint32_t estr[2] = {1, 1};
      r = enc(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      // 16-bit [M][K] as (k % 64, m, k / 64): one box {64, rows, 2} per K block
      const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kStageK), static_cast<cuuint64_t>(M),
                                  static_cast<cuuint64_t>(K / kStageK)};
      const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
      const cuuint32_t box[3] = {static_cast<cuuint32_t>(kStageK), rows, 2};
      const cuuint32_t estr[3] = {1, 1, 1};
      r = enc(&amap,
              pr.mode == kW4A16_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              3, const_cast<void*>(a), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS)
      return fail(W4_ERR_CUDA, "cuTensorMapEncodeTiled (activations) failed (%d)", (int)r);
    static const bool debug = getenv("W4_DEBUG") != nullptr;
    if (debug)
      fprintf(stderr, "w4: %s M=%lld N=%lld K=%lld nj=%d tiles=%d kblocks=%d cluster=%d "
                      "stages=%d grid=%d smem=%zu\n",
              kSchedules[si].name, (long long)M, (long long)N, (long long)K, gp.nj, gp.n_tiles,
              gp.kblocks, gp.cluster, gp.stages, gp.grid, gp.smem_bytes);
    cudaError_t e = launch_gv(gp, amap, args, s);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "gv launch");
  }

  TcPlan plan = make_plan(si, pr.mode, M, N, K, pr.gs);
  args.counters = reinterpret_cast<int*>(ws + plan.ws_counters);
  args.partials = ws + plan.ws_partials;
  args.icopy = reinterpret_cast<int32_t*>(ws + plan.ws_icopy);
  // W4A8 runs on the bf16 copy of its int8 activations in the workspace
  // (staged below, once every tensor map is encoded: an error before that
  // point leaves nothing enqueued)
  const void* act = pr.mode == kW4A8 ? static_cast<const void*>(ws + plan.ws_act) : a;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return fail(W4_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  CUtensorMap amap, smap, zmap;
  memset(&smap, 0, sizeof(smap));
  memset(&zmap, 0, sizeof(zmap));
  const CUtensorMapDataType t16 =
      pr.mode == kW4A16_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (pr.mode == kW4A8F8) {
    // E4M3 [M][K]: one 2-D box of 128 K x BM rows per K block (128-byte rows)
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(plan.bm / (plan.pair ? 2 : 1))};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(act), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(W4_ERR_CUDA, "cuTensorMapEncodeTiled (activations) failed (%d)", (int)r);
    plan.a3d = 0;
  } else {
    // Preferred: one 3-D box {64, BM, nsub} per stage over the view
    // (k % 64, m, k / 64); strides K*2 and 128 bytes.  Fallback: 2-D boxes.
    const cuuint64_t dims3[3] = {static_cast<cuuint64_t>(kStageK), static_cast<cuuint64_t>(M),
                                 static_cast<cuuint64_t>(K / kStageK)};
    const cuuint64_t strides3[2] = {static_cast<cuuint64_t>(K) * 2, 128};
    const cuuint32_t box3[3] = {static_cast<cuuint32_t>(kStageK),
                                static_cast<cuuint32_t>(plan.bm / (plan.pair ? 2 : 1)),
                                static_cast<cuuint32_t>(plan.nsub)};
    const cuuint32_t estr3[3] = {1, 1, 1};
    CUresult r = enc(&amap, t16, 3, const_cast<void*>(act), dims3, strides3, box3, estr3,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    plan.a3d = r == CUDA_SUCCESS ? 1 : 0;
    if (!plan.a3d) {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
      const cuuint32_t box[2] = {static_cast<cuuint32_t>(kStageK),
                                 static_cast<cuuint32_t>(plan.bm / (plan.pair ? 2 : 1))};
      const cuuint32_t estr[2] = {1, 1};
      r = enc(&amap, t16, 2, const_cast<void*>(act), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS)
        return fail(W4_ERR_CUDA, "cuTensorMapEncodeTiled (activations) failed (%d)", (int)r);
    }
  }
  // [G][N] scale / zero-point rows: one box of 128 columns x gps groups per stage
  auto row_map = [&](CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int esz,
                     const char* what) -> w4_status {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / pr.gs)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * esz};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileN), static_cast<cuuint32_t>(plan.gps)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(W4_ERR_CUDA, "cuTensorMapEncodeTiled (%s) failed (%d)", what, (int)r);
    return W4_OK;
  };
  if (b_scales) {
    w4_status st2 = pr.mode == kW4A8
                        ? row_map(&smap, b_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, "group scales")
                        : row_map(&smap, b_scales, t16, 2, "scales");
    if (st2 != W4_OK) return st2;
  }
  if (b_zeros) {
    w4_status st2 = row_map(&zmap, b_zeros, t16, 2, "zero-points");
    if (st2 != W4_OK) return st2;
  }
  static const bool debug = getenv("W4_DEBUG") != nullptr;
  if (debug)
    fprintf(stderr,
            "w4: %s M=%lld N=%lld K=%lld bm=%d nt=%d nsub=%d stages=%d tstages=%d icol=%d gi=%d "
            "acol=%d gps=%d a3d=%d mma2=%d tiles=%d kb=%d grid=%d decomp=%d ksplit=%d segs=%d "
            "smem=%zu\n",
            kSchedules[si].name, (long long)M, (long long)N, (long long)K, plan.bm, plan.nt,
            plan.nsub, plan.stages, plan.tstages, plan.icol, plan.gicopy, plan.acol, plan.gps, plan.a3d,
            tc_mma2(plan) ? 1 : 0, plan.tiles, plan.kb_total, plan.grid, plan.decomp, plan.ksplit,
            plan.max_segs, plan.smem_bytes);
  if (pr.mode == kW4A8 && !prestaged) {
    cudaError_t e = launch_a8_to_bf16(static_cast<const int8_t*>(a), M * K, ws + plan.ws_act, s);
    if (e != cudaSuccess) return cuda_fail(e, "int8->bf16 launch");
  }
  cudaError_t e = launch_tc(plan, amap, smap, zmap, args, s);
  return e == cudaSuccess ? W4_OK : cuda_fail(e, "tc launch");
}

// Workspace of the dynamic-quantization call: the W4A8 GEMM's own, then the
// codes [M][K] and the token scales [M].
struct DynLayout {
  int si;           // schedule of the W4A8 GEMM
  bool prestage;    // tensor-core int8: the quantizer writes the bf16 copy
  size_t gemm_ws, codes, stok, total;
};
DynLayout dyn_layout(int act_type, int64_t M, int64_t N, int64_t K, int64_t gs) {
  DynLayout d{};
  Problem pr{};
  pr.mode = mode_of(act_type);
  pr.M = M;
  pr.N = N;
  pr.K = K;
  pr.gs = gs;
  pr.has_sg = gs != K;
  d.si = default_schedule_impl(pr.mode, M, N, K, gs, pr.has_sg);
  d.prestage = pr.mode == kW4A8 && kSchedules[d.si].engine == kEngineTc && K % 8 == 0 &&
               K <= 32768;
  // the GEMM part always spans the status word and the split-K counters
  // (which every call expects to find zero), whatever its schedule needs
  d.gemm_ws = align256(std::max(ws_needed(d.si, pr), kWsHeader + kCounterBytes));
  d.codes = d.gemm_ws;
  d.stok = align256(d.codes + static_cast<size_t>(M) * K);
  d.total = align256(d.stok + static_cast<size_t>(M) * 4);
  return d;
}

}  // namespace

extern "C" {

size_t w4_gemm_dynamic_workspace_size(int64_t M, int64_t N, int64_t K, int act_type,
                                      int64_t group_size) {
  if (M <= 0 || N <= 0 || K <= 0 || K % kStageK != 0) return kWsHeader;
  if (act_type != W4_S8 && act_type != W4_E4M3) return kWsHeader;
  const int64_t gs = group_size == -1 ? K : group_size;
  if (gs <= 0 || K % gs != 0) return kWsHeader;
  if (act_type == W4_E4M3 && K % 128 != 0) return kWsHeader;
  // the largest over the schedules the call may take (the default one),
  // with room for any schedule an override may name
  const DynLayout d = dyn_layout(act_type, M, N, K, gs);
  const size_t any = w4_gemm_workspace_size(M, N, K, act_type, group_size);
  const size_t extra = d.total - d.gemm_ws;
  return (any > d.gemm_ws ? align256(any) : d.gemm_ws) + extra;
}

w4_status w4_gemm_dynamic(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                          int wtype, int64_t N, const void* b_scales, int scale_type,
                          int64_t group_size, const float* ch_scales, int act_type,
                          const void* bias, void* out, float* token_scales_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 0 || K < 0) return fail(W4_ERR_INVALID_ARGUMENT, "negative size");
  if (a_type != W4_F16 && a_type != W4_BF16)
    return fail(W4_ERR_INVALID_ARGUMENT, "a_type must be W4_F16 or W4_BF16");
  if (act_type != W4_S8 && act_type != W4_E4M3)
    return fail(W4_ERR_INVALID_ARGUMENT, "act_type must be W4_S8 or W4_E4M3");
  if (M == 0 || N == 0) return W4_OK;
  if (K > 0 && !a) return fail(W4_ERR_INVALID_ARGUMENT, "a is null");
  if (!aligned_to(a, 2) || !aligned_to(token_scales_out, 4))
    return fail(W4_ERR_INVALID_ARGUMENT, "a pointer is not aligned to its element size");
  if (K % 8 != 0) return fail(W4_ERR_INVALID_ARGUMENT, "K must be a multiple of 8");
  const int64_t gs = group_size == -1 ? K : group_size;
  if (K > 0 && (gs <= 0 || K % gs != 0))
    return fail(W4_ERR_INVALID_ARGUMENT, "group_size must be -1 or a positive divisor of K");
  if (K == 0 || K % kStageK != 0 || (act_type == W4_E4M3 && K % 128 != 0))
    return fail(W4_ERR_UNSUPPORTED, "K must be a positive multiple of 64 (128 for fp8)");
  if (!workspace || !aligned16(workspace)) return fail(W4_ERR_WORKSPACE, "workspace is null or not 16-byte aligned");
  const DynLayout d = dyn_layout(act_type, M, N, K, gs);
  if (workspace_bytes < d.total)
    return fail(W4_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", workspace_bytes, d.total);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* stok = token_scales_out ? token_scales_out : reinterpret_cast<float*>(ws + d.stok);
  void* codes = ws + d.codes;
  // Check the GEMM's arguments before anything is enqueued (the codes and
  // scales it will read are in the workspace).
  {
    Problem pr{};
    w4_status st = validate(codes, act_type, M, K, b_packed, wtype, N, b_scales, scale_type,
                            nullptr, group_size, stok, ch_scales, out, W4_F16, pr);
    if (st != W4_OK) return st;
    if (bias && !aligned_to(bias, 2))
      return fail(W4_ERR_INVALID_ARGUMENT, "bias is not aligned to its element size");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* qdst = codes;
  int qout = act_type == W4_E4M3 ? 2 : 0;
  // the bf16 form is written from rows held in registers (16-byte loads)
  const bool prestage = d.prestage && aligned16(a);
  if (prestage) {
    const TcPlan plan = make_plan(d.si, kW4A8, M, N, K, gs);
    qdst = ws + plan.ws_act;
    qout = 1;
  }
  cudaError_t e = launch_quant_per_token(a_type == W4_BF16, a, M, K, qdst, stok, qout, s);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return gemm_impl(codes, act_type, M, K, b_packed, wtype, N, b_scales, scale_type, nullptr,
                   group_size, stok, ch_scales, bias, out, W4_F16, workspace, d.gemm_ws, stream,
                   prestage ? d.si : -1, prestage);
}

w4_status w4_gemm_ex(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                     int wtype, int64_t N, const void* b_scales, int scale_type,
                     const void* b_zeros, int64_t group_size, const float* a_token_scales,
                     const float* ch_scales, void* out, int out_type, void* workspace,
                     size_t workspace_bytes, void* stream, int schedule) {
  return gemm_impl(a, a_type, M, K, b_packed, wtype, N, b_scales, scale_type, b_zeros,
                   group_size, a_token_scales, ch_scales, nullptr, out, out_type, workspace,
                   workspace_bytes, stream, schedule);
}

w4_status w4_gemm_bias(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                       int wtype, int64_t N, const void* b_scales, int scale_type,
                       const void* b_zeros, int64_t group_size, const float* a_token_scales,
                       const float* ch_scales, const void* bias, void* out, int out_type,
                       void* workspace, size_t workspace_bytes, void* stream, int schedule) {
  return gemm_impl(a, a_type, M, K, b_packed, wtype, N, b_scales, scale_type, b_zeros,
                   group_size, a_token_scales, ch_scales, bias, out, out_type, workspace,
                   workspace_bytes, stream, schedule);
}

w4_status w4_gemm(const void* a, int a_type, int64_t M, int64_t K, const void* b_packed,
                  int wtype, int64_t N, const void* b_scales, int scale_type,
                  const void* b_zeros, int64_t group_size, const float* a_token_scales,
                  const float* ch_scales, void* out, int out_type, void* workspace,
                  size_t workspace_bytes, void* stream) {
  return w4_gemm_ex(a, a_type, M, K, b_packed, wtype, N, b_scales, scale_type, b_zeros,
                    group_size, a_token_scales, ch_scales, out, out_type, workspace,
                    workspace_bytes, stream, -1);
}

w4_status w4_quantize_per_token(const void* a, int a_type, int64_t M, int64_t K, int8_t* a_q,
                                float* s_tok, void* stream) {
  if (M < 0 || K < 0) return fail(W4_ERR_INVALID_ARGUMENT, "negative size");
  if (a_type != W4_F16 && a_type != W4_BF16)
    return fail(W4_ERR_INVALID_ARGUMENT, "a_type must be W4_F16 or W4_BF16");
  if (M == 0) return W4_OK;
  if (!s_tok || (K > 0 && (!a || !a_q))) return fail(W4_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned_to(a, 2) || !aligned_to(s_tok, 4))
    return fail(W4_ERR_INVALID_ARGUMENT, "a and s_tok must be aligned to their element size");
  if (M > 0x7fffffff) return fail(W4_ERR_UNSUPPORTED, "M above 2^31 - 1");
  cudaError_t e = launch_quant_per_token(a_type == W4_BF16, a, M, K, a_q, s_tok, 0,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4_OK : cuda_fail(e, "quantize launch");
}

w4_status w4_quantize_per_token_fp8(const void* a, int a_type, int64_t M, int64_t K,
                                    uint8_t* a_q, float* s_tok, void* stream) {
  if (M < 0 || K < 0) return fail(W4_ERR_INVALID_ARGUMENT, "negative size");
  if (a_type != W4_F16 && a_type != W4_BF16)
    return fail(W4_ERR_INVALID_ARGUMENT, "a_type must be W4_F16 or W4_BF16");
  if (M == 0) return W4_OK;
  if (!s_tok || (K > 0 && (!a || !a_q))) return fail(W4_ERR_INVALID_ARGUMENT, "null pointer");
  if (!aligned_to(a, 2) || !aligned_to(s_tok, 4))
    return fail(W4_ERR_INVALID_ARGUMENT, "a and s_tok must be aligned to their element size");
  if (M > 0x7fffffff) return fail(W4_ERR_UNSUPPORTED, "M above 2^31 - 1");
  cudaError_t e = launch_quant_per_token(a_type == W4_BF16, a, M, K, a_q, s_tok, 2,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4_OK : cuda_fail(e, "quantize launch");
}

w4_status w4_check_status(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < kWsHeader)
    return fail(W4_ERR_WORKSPACE, "workspace is null or smaller than its header");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word == 0) return W4_OK;
  size_t clear = workspace_bytes < kWsHeader + kCounterBytes ? workspace_bytes
                                                            : kWsHeader + kCounterBytes;
  e = cudaMemset(workspace, 0, clear);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  return fail(W4_ERR_TIMEOUT, "a device-side wait timed out");
}

const char* w4_status_string(int status) {
  switch (status) {
    case W4_OK: return "W4_OK";
    case W4_ERR_INVALID_ARGUMENT: return "W4_ERR_INVALID_ARGUMENT";
    case W4_ERR_UNSUPPORTED: return "W4_ERR_UNSUPPORTED";
    case W4_ERR_WORKSPACE: return "W4_ERR_WORKSPACE";
    case W4_ERR_CUDA: return "W4_ERR_CUDA";
    case W4_ERR_TIMEOUT: return "W4_ERR_TIMEOUT";
    default: return "W4_ERR_UNKNOWN";
  }
}

const char* w4_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
