// api.cu -- the C ABI (include/bi_gemm.h): argument checks, the pin table,
// the launch plan, TMA descriptor encoding, and the launches.
//
// Order of work in every entry point: check every argument (no CUDA call),
// resolve and validate the pins, then touch the device.  A call that returns
// an error has launched nothing.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attention.h"
#include "internal.h"
#include "rowmath.cuh"

#define BI_API extern "C" __attribute__((visibility("default")))

namespace bi {
namespace {

// Fixed design constant used by the default pin table to balance split work
// over a GB300's SMs.  It is never read from the device: the table must not
// depend on anything but (N, K).
constexpr int kTableSmCount = 152;
constexpr int kDefaultSmCount = 152;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The explicit table: the Llama-3.1 projection shapes of the workloads this
// library is measured on.  (N, K) -> (S, T, mma_ctas); mma_ctas 0 leaves the
// CTA grouping to each launch (it never changes a bit).
struct TableEntry {
  int64_t N, K;
  int32_t S, T, ctas;
};
const TableEntry kTable[] = {
    {128, 256, 2, 128, 0},       // tiny invariance shape: exercises the split fold
    {4096, 14336, 4, 256, 0},    // Llama-3.1-8B down_proj: 32 W tiles x 4 = 128 CTAs at decode
    {6144, 4096, 2, 256, 0},     // Llama-3.1-8B qkv: 48 clusters of 2 fit at once (48 of 3 do not)
    {28672, 4096, 2, 256, 0},    // Llama-3.1-8B gate_up: 224 x 2 = 448 (2.95 waves)
    {10240, 8192, 3, 256, 0},    // Llama-3.1-70B qkv: 80 x 3 = 240
    {8192, 8192, 2, 256, 0},     // Llama-3.1-70B o_proj: 64 x 2 = 128
    {57344, 8192, 1, 256, 0},    // Llama-3.1-70B gate_up: 448 tiles, persistent
    {8192, 28672, 2, 256, 0},    // Llama-3.1-70B down_proj: 64 x 2 = 128
};

// Rule for shapes outside the table: the split count that best fills
// kTableSmCount SMs with (N/128) * S equal chains when a whole wave of tiles is
// one token tile (the decode case), with a small charge per extra split.
int32_t rule_split(int64_t N, int64_t K) {
  const int64_t n_tiles = ceil_div(N, kTileN);
  const int64_t kt = ceil_div(K, kBK);
  int32_t best = 1;
  double best_score = -1.0;
  for (int32_t S = 1; S <= 8 && S <= kt; ++S) {
    const int64_t units = n_tiles * S;
    const int64_t waves = ceil_div(units, kTableSmCount);
    const double eff = (double)units / (double)(waves * kTableSmCount);
    const double score = eff - 0.03 * (S - 1);
    if (score > best_score + 1e-12) {
      best_score = score;
      best = S;
    }
  }
  return best;
}

// Operand type of a GEMM.  A K tile is 128 bytes of a row either way: 64 bf16
// or 128 E4M3 values.
enum class Elem { BF16, E4M3 };
constexpr int tile_elems(Elem e) { return e == Elem::E4M3 ? 128 : kBK; }
constexpr int elem_bytes(Elem e) { return e == Elem::E4M3 ? 1 : 2; }

// K must give 16-byte rows (the tensor-memory copies' row pitch).
bi_status check_nk(int64_t N, int64_t K, Elem e = Elem::BF16) {
  if (N < 1 || K < 1) return BI_ERR_INVALID_ARG;
  if ((K * elem_bytes(e)) % 16 != 0) return BI_ERR_UNSUPPORTED_SHAPE;
  if (N > 0x7FFFFFFFll || K > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  return BI_OK;
}

struct Resolved {
  int32_t S, T, ctas, w_pin;
  uint32_t flags;
  int64_t KT, K;
  Elem elem;
};

// K tiles per copy for a launch with token tile T and CTA grouping ctas: 2
// when the flag asks for it and it is possible (K % 64 == 0, T = 256, or a
// narrower paired tile of 224, 192 or 160) and the MMAs are paired, else 1.
// (A single CTA at T = 256 has a 48 KB K tile; its rings would hold only two
// X stages of two tiles, which measured slower.)  Otherwise, launches whose X
// copies cover fewer rows than the token tile use 1, except decode tiles on
// single-CTA MMAs, which take two K tiles per stage by 2-D copies
// (make_plan).
int pins_kps(int64_t K, int32_t T, int32_t ctas, uint32_t flags, Elem e = Elem::BF16) {
  const bool wide = T == 256 || T == 224 || T == 192 || T == 160;
  return ((flags & BI_FLAG_KTILE_PAIRS) && K % tile_elems(e) == 0 && wide && ctas == 2) ? 2 : 1;
}

bi_status resolve_pins(int64_t N, int64_t K, const bi_pins* pins, Resolved* r, Elem e = Elem::BF16);

// Which device function pointer encodes tensor maps (driver entry point).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A [rows, K] bf16 row-major matrix, 128-byte swizzle, zero fill outside the
// matrix.  view3d false: a 2-D map, box 64 x box_rows (one K tile, kps 1).
// view3d true (K % 64 == 0 only): the same bytes seen as [K/64][rows][64], box
// 64 x box_rows x kps, so one copy lands kps K tiles one after another in
// shared memory, each box_rows x 128 bytes.  Without K % 64 == 0 the 3-D view
// would read a partial last K tile's tail from the next row instead of zeros.
bool encode_kmajor(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int box_rows,
                   bool view3d, int kps, Elem e = Elem::BF16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const CUtensorMapDataType dt = e == Elem::E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t te = tile_elems(e), eb = elem_bytes(e);
  CUresult r;
  if (!view3d) {
    if (kps != 1) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K * eb)};
    cuuint32_t box[2] = {(cuuint32_t)te, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    r = enc(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    if (K % te != 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)te, (cuuint64_t)rows, (cuuint64_t)(K / te)};
    cuuint64_t strides[2] = {(cuuint64_t)(K * eb), (cuuint64_t)(te * eb)};
    cuuint32_t box[3] = {(cuuint32_t)te, (cuuint32_t)box_rows, (cuuint32_t)kps};
    cuuint32_t estr[3] = {1, 1, 1};
    r = enc(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

int sm_count_current() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kDefaultSmCount;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = kDefaultSmCount;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

// Clusters of `size` CTAs that can be resident at once, at one CTA per SM.
// Measured on GB300 (152 SMs, about 231 KB of shared memory per CTA): 76 of
// 2, 36 of 4, 23 of 6, 15 of 8 -- a cluster must fit in one GPC.  Elsewhere
// an estimate.  Speed only.
int64_t max_clusters(int32_t size, int32_t sm_count) {
  if (size <= 1) return sm_count;
  if (sm_count == kDefaultSmCount) {
    switch (size) {
      case 2: return 76;
      case 4: return 36;
      case 6: return 23;
      case 8: return 15;
      default: break;
    }
  }
  const double est = (double)sm_count / size * (1.0 - size / 40.0);
  return est < 1.0 ? 1 : (int64_t)est;
}

struct LaunchChoice {
  int32_t ctas, schedule, units;
  double cost;
  int32_t T = 0;  // token tile of the launch (0: the pinned one)
};

// Best schedule for one CTA grouping, and its cost in units of one K tile of a
// paired MMA (about 0.33 us on GB300), calibrated on down_proj launches:
//   - a one-CTA K tile (half the W rows) costs 1.2 pair K tiles: its operands
//     are 48 KB per K tile against 32 KB for each CTA of a pair;
//   - a cluster wave adds about 30 K tiles (pipeline fill, the epilogue that
//     no other chain overlaps, the fold); a persistent launch about 15.
//   LOCAL   ceil(tiles / units) tiles of S chains per persistent unit;
//   CLUSTER waves of resident S-unit clusters, one chain per unit;
//   CHAIN   waves of resident ceil(S/2)-unit clusters, two chains per unit.
// A single short token tile (decode) streams W from HBM: there the schedule
// that puts the most CTAs on the W stream wins, which the rounds of LOCAL
// against those of CLUSTER capture (CHAIN is not used).
// GLOBAL (a fold workspace at hand, one token tile, single-CTA MMAs,
// 2 <= S <= BI_GLOBAL_MAX_SPLIT_K): rounds of ceil(tiles * S / SMs) chains on
// persistent CTAs, with no co-residency limit.
LaunchChoice best_schedule(const Resolved& r, int32_t ctas, int64_t M, int64_t N, int32_t sm_count,
                           bool fold_ok) {
  const uint32_t forced = r.flags & BI_FLAG_SCHEDULE_MASK;
  const int64_t n_tiles = ceil_div(N, (int64_t)kTileN * ctas);
  const int64_t m_tiles = ceil_div(M, r.T);
  const int64_t tiles = n_tiles * m_tiles;
  const bool grid_ok = n_tiles <= 65535 && m_tiles <= 65535;
  const int32_t uc = (r.S + 1) / 2;
  const int64_t slots = sm_count / ctas > 0 ? sm_count / ctas : 1;
  const double k = ctas == 2 ? 1.0 : 1.2;          // cost of one K tile
  const double chain = (double)r.KT / r.S * k;      // one split chain
  LaunchChoice local{ctas, BI_FLAG_SCHEDULE_LOCAL, 1,
                     (double)ceil_div(tiles, slots) * r.S * chain + 15.0};
  LaunchChoice cl{ctas, BI_FLAG_SCHEDULE_CLUSTER, r.S,
                  (double)ceil_div(tiles, max_clusters(r.S * ctas, sm_count)) * (chain + 30.0)};
  LaunchChoice ch{ctas, BI_FLAG_SCHEDULE_CHAIN, uc,
                  (double)ceil_div(tiles, max_clusters(uc * ctas, sm_count)) * (2.0 * chain + 30.0)};
  const bool global_ok = fold_ok && ctas == 1 && m_tiles == 1 && r.S >= 2 && r.S <= BI_GLOBAL_MAX_SPLIT_K &&
                         tiles * r.S <= 0x7FFFFFFF;
  const LaunchChoice gl{ctas, BI_FLAG_SCHEDULE_GLOBAL, 1, 0.0};
  if (r.S == 1 || forced == BI_FLAG_SCHEDULE_LOCAL || !grid_ok) return local;
  if (forced == BI_FLAG_SCHEDULE_CLUSTER) return cl;
  if (forced == BI_FLAG_SCHEDULE_CHAIN) return ch;
  if (forced == BI_FLAG_SCHEDULE_GLOBAL && global_ok) return gl;
  if (m_tiles == 1 && M <= r.T / 2) {
    // decode: rounds of chain work per unit.  CLUSTER runs in waves of the
    // clusters that fit at once, charged 15%; GLOBAL spreads the chains over
    // every SM, but its fold through L2 costs more than one DSMEM fold
    // (measured on GB300: 1-2 us at M = 32), so it is taken where it runs
    // fewer rounds than the clusters' waves, or where the clusters need
    // several waves (each wave pays its start and its fold; Llama-3.1-8B
    // gate_up at decode: 3 waves in 47 us, 3 GLOBAL rounds in 38 us).
    const double local_rounds = (double)ceil_div(tiles, slots) * r.S;
    const int64_t waves = r.S * ctas <= 8 ? ceil_div(tiles, max_clusters(r.S * ctas, sm_count)) : INT64_MAX;
    const double cluster_rounds = waves == INT64_MAX ? 1e30 : (double)waves * 1.15;
    const int64_t rounds = global_ok ? ceil_div(tiles * r.S, sm_count) : INT64_MAX;
    if (rounds != INT64_MAX && (rounds < waves || (waves > 1 && rounds <= waves)) && (double)rounds <= local_rounds)
      return gl;
    return cluster_rounds < local_rounds ? cl : local;
  }
  LaunchChoice best = local;
  if (r.S * ctas <= 8 && cl.cost < best.cost) best = cl;
  if (r.S >= 3 && uc * ctas <= 8 && ch.cost < best.cost) best = ch;
  return best;
}

// The CTA grouping (when the pins leave it open, mma_ctas = 0) and the
// schedule, from M.  cta_group::1 and ::2 MMAs give every output element the
// same bits (each element is one chain of k16 steps in the same order on
// either SM of a pair; tested on GPU), so this is speed only.  A single short
// token tile (M <= T/2) stays on one CTA per MMA: a pair would hold a
// half-empty X box, and decode is bound by the W stream, which S-CTA clusters
// spread over the most SMs.  A forced one-split CLUSTER schedule also keeps
// one CTA (a pair would need clusters of 2S).
LaunchChoice choose_launch(int64_t M, int64_t N, const Resolved& r, int32_t sm_count, bool fold_ok) {
  if (r.ctas != 0) return best_schedule(r, r.ctas, M, N, sm_count, fold_ok);
  const LaunchChoice one = best_schedule(r, 1, M, N, sm_count, fold_ok);
  if (M <= r.T / 2 || (r.flags & BI_FLAG_SCHEDULE_MASK) == BI_FLAG_SCHEDULE_CLUSTER) return one;
  LaunchChoice two = best_schedule(r, 2, M, N, sm_count, fold_ok);
  // A persistent paired launch may also narrow its token tile so that the
  // tiles fill the last wave (224, 192 or 160 instead of 256).  Its per-K-tile
  // cost follows the operand bytes each CTA receives: 16 KB of W and T/2 rows
  // of X, against 32 KB at T = 256 (the MMA itself takes T/2 of its 128
  // cycles, within that).
  if (two.schedule == BI_FLAG_SCHEDULE_LOCAL && r.T == 256 && r.elem == Elem::BF16 &&
      pins_kps(r.K, 256, 2, r.flags) == 2 && M > r.T / 2) {
    const int64_t n_tiles = ceil_div(N, (int64_t)kTileN * 2);
    const int64_t slots = sm_count / 2 > 0 ? sm_count / 2 : 1;
    for (int32_t t : {224, 192, 160}) {
      const double k = (16.0 + t / 16.0) / 32.0;
      const double cost = (double)ceil_div(n_tiles * ceil_div(M, (int64_t)t), slots) * (double)r.KT * k + 15.0;
      if (cost < two.cost * 0.98) {
        two.cost = cost;
        two.T = t;
      }
    }
  }
  return two.cost < one.cost ? two : one;
}

// Fold workspace bytes of a GLOBAL plan: the per-tile arrival counters
// (rounded up to 256 bytes), then the chain partials [tiles * S][T][128] fp32.
size_t fold_bytes(const bi_gemm_plan& plan) {
  const uint64_t tiles = (uint64_t)plan.n_tiles * (uint64_t)plan.m_tiles;
  const uint64_t counters = (tiles * 4u + 255u) & ~(uint64_t)255u;
  return (size_t)(counters + tiles * (uint64_t)plan.split_k * (uint64_t)plan.tok_tile * kTileN * 4u);
}

bi_status make_plan_once(int64_t M, int64_t N, int64_t K, const Resolved& pinned, int32_t sm_count, bool fold_ok,
                         bi_gemm_plan* plan) {
  std::memset(plan, 0, sizeof(*plan));
  Resolved r = pinned;
  const LaunchChoice choice = choose_launch(M, N, r, sm_count, fold_ok);
  r.ctas = choice.ctas;
  if (choice.T != 0) r.T = choice.T;
  // Decode (M <= 128 on single-CTA MMAs, the CTA grouping and the W depth
  // left open by the pins; bf16 or E4M3): the token tile narrows to 64 or
  // 128, whichever holds M (the MMA's N extent changes no bit), and W and X
  // come two K tiles per stage by two 2-D copies each.  W streams from HBM
  // faster in stages of 256 bytes per row than of 128 (5.5 against 4.1 TB/s
  // measured for the down_proj pattern), and the narrower X stages leave the
  // shared memory to them.  (At T = 256 the same stages leave room for only
  // 3 W and 2 X stages, which measured slower: 34.3 against 30.9 us for
  // down_proj at M = 256.)
  const bool decode2 = pinned.ctas == 0 && r.ctas == 1 && M > 0 && M <= 128 && M <= r.T && r.w_pin == 0 &&
                       (r.flags & BI_FLAG_KTILE_PAIRS) != 0;
  if (decode2) r.T = M <= 64 ? 64 : 128;
  plan->bk = tile_elems(r.elem);
  plan->split_k = r.S;
  plan->tok_tile = r.T;
  plan->mma_ctas = r.ctas;
  plan->mma_m = kTileN * r.ctas;
  plan->mma_n = r.T;
  plan->mma_k = r.elem == Elem::E4M3 ? 2 * kMmaK : kMmaK;
  plan->k_tiles = r.KT;
  for (int s = 0; s <= r.S; ++s) plan->split_begin[s] = ((int64_t)s * r.KT) / r.S;
  plan->n_tiles = ceil_div(N, plan->mma_m);
  plan->m_tiles = M > 0 ? ceil_div(M, r.T) : 0;
  // Token rows each CTA holds per X stage, and how many of them a copy brings
  // in: a single token tile loads only its valid rows (rounded up to 8); the
  // rest of each X stage is zeroed once and never rewritten.  Speed only: the
  // MMA still reads all rows, and rows past M are zero either way.
  const int32_t x_rows = r.T / r.ctas;
  plan->x_box_rows = (plan->m_tiles == 1 && M <= x_rows) ? (int32_t)((M + 7) / 8 * 8) : x_rows;
  if (plan->x_box_rows > x_rows) plan->x_box_rows = x_rows;
  // a short X box keeps one K tile per copy: each K tile of X must start
  // x_rows rows after the previous one in shared memory
  plan->kps = decode2 ? 2 : (plan->x_box_rows == x_rows ? pins_kps(K, r.T, r.ctas, r.flags, r.elem) : 1);
  choose_stages(x_rows, plan->x_box_rows, r.w_pin, plan->kps, &plan->w_stages, &plan->x_stages);
  plan->block_threads = kGemmThreads;
  const int64_t tiles = plan->n_tiles * plan->m_tiles;
  plan->schedule = choice.schedule;
  plan->units = choice.units;
  const bool cluster = plan->schedule == BI_FLAG_SCHEDULE_CLUSTER || plan->schedule == BI_FLAG_SCHEDULE_CHAIN;
  if (plan->schedule == BI_FLAG_SCHEDULE_GLOBAL) {
    const int64_t chains = tiles * r.S;
    plan->grid_x = (int32_t)(chains < sm_count ? chains : sm_count);
    plan->grid_y = 1;
    plan->grid_z = 1;
    plan->cluster_x = 1;
    plan->group_n = 1;
  } else if (cluster) {
    if (plan->n_tiles > 65535 || plan->m_tiles > 65535) return BI_ERR_UNSUPPORTED_SHAPE;
    plan->grid_x = choice.units * r.ctas;
    plan->grid_y = (int32_t)plan->n_tiles;
    plan->grid_z = (int32_t)plan->m_tiles;
    plan->cluster_x = choice.units * r.ctas;
  } else {
    const int64_t slots = sm_count / r.ctas > 0 ? sm_count / r.ctas : 1;
    const int64_t units = tiles < slots ? tiles : slots;
    plan->grid_x = (int32_t)(units * r.ctas);
    plan->grid_y = 1;
    plan->grid_z = 1;
    plan->cluster_x = r.ctas;
    // about sqrt(units) W tiles per group: the units in flight then cover as
    // many W tiles as token tiles
    int64_t g = 1;
    while ((g + 1) * (g + 1) <= units) ++g;
    plan->group_n = (int32_t)(g < plan->n_tiles ? g : plan->n_tiles);
  }
  plan->smem_bytes = gemm_smem_bytes(r.T, x_rows, plan->w_stages, plan->x_stages, plan->kps, cluster);
  if (plan->w_stages < 2 || plan->x_stages < 2) return BI_ERR_ILLEGAL_PINS;
  if (plan->smem_bytes > kMaxDynSmem) return BI_ERR_ILLEGAL_PINS;
  return BI_OK;
}

// The plan for a call with `fold_avail` bytes of fold workspace: GLOBAL only
// where the planner picks it and its workspace fits.
bi_status make_plan(int64_t M, int64_t N, int64_t K, const Resolved& pinned, int32_t sm_count,
                    bi_gemm_plan* plan, size_t fold_avail = 0) {
  bi_status st = make_plan_once(M, N, K, pinned, sm_count, fold_avail > 0, plan);
  if (st == BI_OK && plan->schedule == BI_FLAG_SCHEDULE_GLOBAL && fold_bytes(*plan) > fold_avail)
    st = make_plan_once(M, N, K, pinned, sm_count, false, plan);
  return st;
}

bi_status validate(int64_t N, int64_t K, const bi_pins* p, Elem e = Elem::BF16) {
  if (!p) return BI_ERR_INVALID_ARG;
  bi_status st = check_nk(N, K, e);
  if (st != BI_OK) return st;
  const int64_t kt = ceil_div(K, tile_elems(e));
  if (p->abi_version != BI_PINS_ABI_VERSION) return BI_ERR_ILLEGAL_PINS;
  if (p->bk != tile_elems(e)) return BI_ERR_ILLEGAL_PINS;
  if (e == Elem::E4M3 && p->tok_tile != 256) return BI_ERR_ILLEGAL_PINS;
  if (p->split_k < 1 || p->split_k > BI_MAX_SPLIT_K || p->split_k > kt) return BI_ERR_ILLEGAL_PINS;
  if (p->tok_tile != 64 && p->tok_tile != 128 && p->tok_tile != 256) return BI_ERR_ILLEGAL_PINS;
  if (p->mma_ctas < 0 || p->mma_ctas > 2) return BI_ERR_ILLEGAL_PINS;
  // a W depth must leave two X stages at the largest copies of every CTA
  // grouping the pins allow
  if (p->stages != 0) {
    if (p->stages < 2) return BI_ERR_ILLEGAL_PINS;
    for (int32_t ctas = 1; ctas <= 2; ++ctas) {
      if (p->mma_ctas != 0 && p->mma_ctas != ctas) continue;
      const int kps = pins_kps(K, p->tok_tile, ctas, p->flags, e);
      if (p->stages > max_w_stages(p->tok_tile / ctas, 2, kps)) return BI_ERR_ILLEGAL_PINS;
    }
  }
  if (p->flags & ~BI_FLAG_KNOWN_MASK) return BI_ERR_ILLEGAL_PINS;
  if ((p->flags & BI_FLAG_NORM_SMEM) && (p->flags & BI_FLAG_NORM_STAGED)) return BI_ERR_ILLEGAL_PINS;
  const uint32_t sched = p->flags & BI_FLAG_SCHEDULE_MASK;
  if (sched == BI_FLAG_SCHEDULE_CLUSTER && p->split_k * (p->mma_ctas == 2 ? 2 : 1) > 16)
    return BI_ERR_ILLEGAL_PINS;
  if (sched == BI_FLAG_SCHEDULE_CLUSTER && p->split_k > 8) return BI_ERR_ILLEGAL_PINS;
  if (sched > BI_FLAG_SCHEDULE_GLOBAL) return BI_ERR_ILLEGAL_PINS;
  // CHAIN: ceil(S/2) >= 2 units per tile; an open grouping may choose pairs
  if (sched == BI_FLAG_SCHEDULE_CHAIN &&
      (p->split_k < 3 || (p->split_k + 1) / 2 * (p->mma_ctas == 1 ? 1 : 2) > 16))
    return BI_ERR_ILLEGAL_PINS;
  return BI_OK;
}

bi_status pins_default(int64_t N, int64_t K, bi_pins* out, Elem e = Elem::BF16) {
  if (!out) return BI_ERR_INVALID_ARG;
  bi_status st = check_nk(N, K, e);
  if (st != BI_OK) return st;
  int32_t S = 0, T = 256, ctas = 0;
  for (const TableEntry& e : kTable) {
    if (e.N == N && e.K == K) {
      S = e.S;
      T = e.T;
      ctas = e.ctas;
      break;
    }
  }
  if (S == 0) S = rule_split(N, K);
  const int64_t kt = ceil_div(K, tile_elems(e));
  if (S > kt) S = (int32_t)kt;
  if (e == Elem::E4M3) T = 256;
  out->abi_version = BI_PINS_ABI_VERSION;
  out->bk = tile_elems(e);
  out->split_k = S;
  out->tok_tile = T;
  out->mma_ctas = ctas;
  out->stages = 0;
  out->flags = BI_FLAG_SCHEDULE_AUTO | BI_FLAG_KTILE_PAIRS;
  return BI_OK;
}

bi_status resolve_pins(int64_t N, int64_t K, const bi_pins* pins, Resolved* r, Elem e) {
  bi_pins p;
  if (pins) {
    p = *pins;
  } else {
    bi_status st = pins_default(N, K, &p, e);
    if (st != BI_OK) return st;
  }
  bi_status st = validate(N, K, &p, e);
  if (st != BI_OK) return st;
  r->S = p.split_k;
  r->T = p.tok_tile;
  r->ctas = p.mma_ctas;
  r->w_pin = p.stages;
  r->flags = p.flags;
  r->KT = ceil_div(K, tile_elems(e));
  r->K = K;
  r->elem = e;
  return BI_OK;
}

bi_status check_rmsnorm_args(const void* X, const void* g, const void* Y, int64_t M, int64_t H,
                             float eps) {
  if (M < 0 || H < 1) return BI_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || !(eps < 3.0e38f)) return BI_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > 65536) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!X || !g || !Y) return BI_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(g) || !aligned16(Y)) return BI_ERR_ALIGNMENT;
  return BI_OK;
}

bi_status check_gemm_args(const void* X, const void* W, const void* Y, int64_t M, int64_t N,
                          int64_t K, Elem e = Elem::BF16) {
  if (M < 0) return BI_ERR_INVALID_ARG;
  bi_status st = check_nk(N, K, e);
  if (st != BI_OK) return st;
  if (M > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!X || !W || !Y) return BI_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Y)) return BI_ERR_ALIGNMENT;
  return BI_OK;
}

// Step 1 of a GEMM launch: argument checks, pins and the plan, with no CUDA
// call.  L->M == 0 means there is nothing to launch.
bi_status plan_gemm(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                    const bi_pins* pins, cudaStream_t stream, GemmLaunch* out, Elem e = Elem::BF16,
                    const float* sx = nullptr, const float* sw = nullptr, void* fold_ws = nullptr,
                    size_t fold_avail = 0) {
  bi_status st = check_gemm_args(X, W, Y, M, N, K, e);
  if (st != BI_OK) return st;
  if (e == Elem::E4M3 && M > 0) {
    if (!sx || !sw) return BI_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(sx) & 3u) || (reinterpret_cast<uintptr_t>(sw) & 3u)) return BI_ERR_ALIGNMENT;
  }
  Resolved r;
  st = resolve_pins(N, K, pins, &r, e);
  if (st != BI_OK) return st;
  GemmLaunch& L = *out;
  std::memset(&L, 0, sizeof(L));
  if (M == 0) return BI_OK;
  bi_gemm_plan plan;
  st = make_plan(M, N, K, r, sm_count_current(), &plan, fold_ws ? fold_avail : 0);
  if (st != BI_OK) return st;
  if (plan.schedule == BI_FLAG_SCHEDULE_GLOBAL) {
    const uint64_t tiles = (uint64_t)plan.n_tiles * (uint64_t)plan.m_tiles;
    L.fold_count = static_cast<uint32_t*>(fold_ws);
    L.fold_part = reinterpret_cast<float*>(static_cast<char*>(fold_ws) + ((tiles * 4u + 255u) & ~(uint64_t)255u));
  }
  L.X = X;
  L.W = W;
  L.fp8 = e == Elem::E4M3;
  L.sx = sx;
  L.sw = sw;
  L.Y = Y;
  L.M = M;
  L.N = N;
  L.K = K;
  L.n_tiles = (int32_t)plan.n_tiles;
  L.m_tiles = (int32_t)plan.m_tiles;
  L.k_tiles = (int32_t)r.KT;
  L.S = r.S;
  L.T = plan.tok_tile;  // the launch's token tile (may be narrower than the pinned one)
  L.w_stages = plan.w_stages;
  L.x_stages = plan.x_stages;
  L.x_box_rows = plan.x_box_rows;
  L.kps = plan.kps;
  L.group_n = plan.group_n > 0 ? plan.group_n : 1;
  L.units = plan.units;
  L.cluster = plan.schedule == BI_FLAG_SCHEDULE_CLUSTER || plan.schedule == BI_FLAG_SCHEDULE_CHAIN;
  L.pair = plan.mma_ctas == 2;
  L.grid_x = plan.grid_x;
  L.grid_y = plan.grid_y;
  L.grid_z = plan.grid_z;
  L.smem = plan.smem_bytes;
  L.flags = r.flags;
  // two K tiles per copy (3-D maps) on paired MMAs; single-CTA MMAs with two
  // K tiles per stage take them as two 2-D copies
  if (plan.kps > 1 && plan.mma_ctas == 1) L.flags |= kFlagCopy2D;
  if (plan.x_box_rows < plan.tok_tile / plan.mma_ctas) L.flags |= kFlagZeroX;
  if (plan.m_tiles == 1) L.flags |= kFlagStreamW;
#ifdef BI_DEBUG_BOUNDS
  {
    const char* poke = std::getenv("BI_DEBUG_POKE");
    if (poke && std::strcmp(poke, "wrow") == 0) L.flags |= kFlagDebugPokeWRow;
  }
#endif
  L.stream = stream;
  return BI_OK;
}

// Step 2: the tensor maps and the status word (driver calls, no launch).
bi_status encode_gemm(GemmLaunch& L) {
  const Elem e = L.fp8 ? Elem::E4M3 : Elem::BF16;
  const bool map3d = L.kps > 1 && !(L.flags & kFlagCopy2D);
  if (!encode_kmajor(&L.tmW, L.W, L.N, L.K, kTileN, map3d, map3d ? L.kps : 1, e)) return BI_ERR_CUDA;
  if (!encode_kmajor(&L.tmX, L.X, L.M, L.K, L.x_box_rows, map3d, map3d ? L.kps : 1, e)) return BI_ERR_CUDA;
  L.status = device_status_word();
  if (!L.status) return BI_ERR_CUDA;
  return BI_OK;
}

}  // namespace

// The RMSNorm -> GEMM layer, checked and planned (no CUDA call): X [M,K] raw
// activations, g [K], W [N,K], Y [M,N].
bi_status plan_fused(const void* X, const void* g, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                     float eps, const bi_pins* pins, cudaStream_t stream, GemmLaunch* L, void* fold_ws,
                     size_t fold_avail) {
  bi_status st = check_gemm_args(X, W, Y, M, N, K);
  if (st != BI_OK) return st;
  st = check_rmsnorm_args(X, g, Y, M, K, eps);
  if (st != BI_OK) return st;
  st = plan_gemm(X, W, Y, M, N, K, pins, stream, L, Elem::BF16, nullptr, nullptr, fold_ws, fold_avail);
  if (st != BI_OK) return st;
  L->g = g;
  L->eps = eps;
  return BI_OK;
}

// The staged form unless the pins force shared memory: measured faster on
// GB300 at every batch size of the Llama-3.1-8B projections.
bool fused_in_smem(const GemmLaunch& L) { return (L.flags & BI_FLAG_NORM_SMEM) != 0; }

size_t fused_r_bytes(int64_t M) { return (size_t)(((uint64_t)M * 4u + 255u) & ~(uint64_t)255u); }

size_t fused_staged_bytes(int64_t M, int64_t K) {
  return (size_t)(((uint64_t)M * (uint64_t)K * 2u + 255u) & ~(uint64_t)255u);
}

size_t fused_workspace_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0) return 0;
  return fused_r_bytes(M) + fused_staged_bytes(M, K);
}

// Encodes the planned layer's tensor maps, then launches it.  In shared
// memory: the row-scale kernel (r[m] of every row into the workspace's
// first part) and the GEMM that normalises X in shared memory with it.
// Staged: the RMSNorm kernel writes the normalised rows to the workspace's
// second part and the GEMM reads them.  An encoding failure returns before
// the first launch.
bi_status launch_fused(GemmLaunch& L, void* ws, bool in_smem) {
  if (L.M == 0) return BI_OK;
  const void* X = L.X;
  if (!in_smem) L.X = static_cast<char*>(ws) + fused_r_bytes(L.M);
  bi_status st = encode_gemm(L);
  if (st != BI_OK) return st;
  if (!in_smem) {
    if (launch_rmsnorm(X, L.g, const_cast<void*>(L.X), L.M, L.K, L.eps, L.stream) != cudaSuccess)
      return BI_ERR_CUDA;
    return launch_gemm(L) == cudaSuccess ? BI_OK : BI_ERR_CUDA;
  }
  if (L.M <= kRowScaleInKernelMax && L.m_tiles == 1) {
    L.rrow = nullptr;  // the GEMM computes the few rows' r itself: one launch
    return launch_gemm_fused(L) == cudaSuccess ? BI_OK : BI_ERR_CUDA;
  }
  float* r = static_cast<float*>(ws);
  L.rrow = r;
  if (launch_row_scale(X, r, L.M, L.K, L.eps, L.stream) != cudaSuccess) return BI_ERR_CUDA;
  return launch_gemm_fused(L) == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

namespace {

bi_status gemm_impl(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                    const bi_pins* pins, cudaStream_t stream, Elem e = Elem::BF16,
                    const float* sx = nullptr, const float* sw = nullptr, void* fold_ws = nullptr,
                    size_t fold_avail = 0) {
  GemmLaunch L;
  bi_status st = plan_gemm(X, W, Y, M, N, K, pins, stream, &L, e, sx, sw, fold_ws, fold_avail);
  if (st != BI_OK || L.M == 0) return st;
  st = encode_gemm(L);
  if (st != BI_OK) return st;
  return launch_gemm(L) == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

// ---- the GEMM on host buffers: rows in chunks through a ring of device buffers
//
// Chunk c's rows are copied in on one stream, multiplied on the caller's
// stream and copied out on another, so the copies of one chunk overlap the
// GEMM of the next.  Batch invariance makes this free: a row's bits do not
// depend on the chunk (the M of the launch) it travels in.  A list of jobs of
// one (N, K) runs as one sequence of chunks, so the copies of one job overlap
// the GEMMs of its neighbours too.
constexpr int kHostSlots = 2;     // ring depth of the workspace size the query returns
constexpr int kHostMaxSlots = 8;  // deepest ring a larger workspace buys

int64_t host_chunk_rows(int64_t M, int64_t K) {
  int64_t r = (int64_t{16} << 20) / (2 * K);  // about 16 MB of X per chunk
  r = r / 128 * 128;
  r = r < 128 ? 128 : (r > 8192 ? 8192 : r);
  return r < M ? r : M;
}

uint64_t round256(uint64_t b) { return (b + 255u) & ~(uint64_t)255u; }

// bytes of one ring slot: the chunk's X, then its Y
uint64_t host_slot_bytes(int64_t R, int64_t N, int64_t K) {
  return round256((uint64_t)R * (uint64_t)K * 2u) + round256((uint64_t)R * (uint64_t)N * 2u);
}

// Chunk rows R (chunk_rows, else the rule above for the largest job, and at
// most the largest job's rows) and the number of chunks of all jobs; false for
// a negative or oversized M or chunk_rows.
bool host_chunking(const bi_host_gemm_job* jobs, int32_t n, int64_t K, int64_t chunk_rows, int64_t* R,
                   int64_t* chunks) {
  if (chunk_rows < 0 || chunk_rows > 0x7FFFFFFFll) return false;
  int64_t mmax = 0;
  for (int32_t j = 0; j < n; ++j) {
    if (jobs[j].M < 0 || jobs[j].M > 0x7FFFFFFFll) return false;
    mmax = jobs[j].M > mmax ? jobs[j].M : mmax;
  }
  *R = chunk_rows > 0 ? (chunk_rows < mmax ? chunk_rows : mmax) : host_chunk_rows(mmax, K);
  *chunks = 0;
  for (int32_t j = 0; j < n; ++j)
    if (jobs[j].M > 0) *chunks += (jobs[j].M + *R - 1) / *R;
  return true;
}

// Rows of the next chunk when `left` rows of a job remain: R, except that
// the list's last rows go in halving chunks (half the rows left, rounded down
// to a multiple of 128, at least 128; the last 256 rows or fewer whole), so
// that what is left after the last copy-in -- that chunk's GEMM and its
// copy-out -- is short.  Only with a ring of three or more slots (measured on
// the down_proj sweep as one list: 2.507 against 2.599 ms with 8 slots; one
// call per M with 2 slots lost 2%).
constexpr int64_t kHostTaperRows = 128;

int64_t host_next_rows(int64_t left, int64_t R, bool taper) {
  if (!taper || left > 2 * R || left <= 2 * kHostTaperRows) return left < R ? left : R;
  int64_t half = left / 2 / kHostTaperRows * kHostTaperRows;
  half = half < kHostTaperRows ? kHostTaperRows : half;
  return half < R ? half : R;
}

size_t host_workspace_bytes(const bi_host_gemm_job* jobs, int32_t n, int64_t N, int64_t K, int64_t chunk_rows) {
  if (n <= 0 || !jobs || N <= 0 || K <= 0) return 0;
  int64_t R = 0, chunks = 0;
  if (!host_chunking(jobs, n, K, chunk_rows, &R, &chunks) || chunks == 0) return 0;
  return (size_t)((chunks < kHostSlots ? chunks : kHostSlots) * host_slot_bytes(R, N, K));
}

// Per-device streams and events, created once and reused by every call; a
// per-device mutex keeps one call's enqueue sequence whole.
struct HostCtx {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t copied_in[kHostMaxSlots] = {}, multiplied[kHostMaxSlots] = {}, copied_out[kHostMaxSlots] = {};
  bool ready = false;
};
HostCtx g_host_ctx[64];
std::mutex g_host_mu[64];

bool host_ctx_init(HostCtx& c) {
  if (c.ready) return true;
  const unsigned ef = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&c.start, ef) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&c.end, ef) != cudaSuccess) return false;
  for (int i = 0; i < kHostMaxSlots; ++i) {
    if (cudaEventCreateWithFlags(&c.copied_in[i], ef) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&c.multiplied[i], ef) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&c.copied_out[i], ef) != cudaSuccess) return false;
  }
  c.ready = true;
  return true;
}

// The checks the call and its schedule query share: the list, the rows, the
// shape and chunk_rows.  Sets R and the chunk count before the taper.
bi_status host_check_rows(const bi_host_gemm_job* jobs, int32_t n, int64_t N, int64_t K, int64_t chunk_rows,
                          int64_t* R, int64_t* chunks) {
  if (n < 0 || (n > 0 && !jobs) || chunk_rows < 0) return BI_ERR_INVALID_ARG;
  for (int32_t j = 0; j < n; ++j)
    if (jobs[j].M < 0) return BI_ERR_INVALID_ARG;
  bi_status st = check_nk(N, K);
  if (st != BI_OK) return st;
  for (int32_t j = 0; j < n; ++j)
    if (jobs[j].M > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  if (chunk_rows > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  *R = 0;
  *chunks = 0;
  host_chunking(jobs, n, K, chunk_rows, R, chunks);
  return BI_OK;
}

// Ring depth: as many slots as the workspace holds, up to kHostMaxSlots and
// the chunk count.
int64_t host_depth(size_t ws_bytes, uint64_t slot, int64_t chunks) {
  int64_t depth = (int64_t)(ws_bytes / slot);
  depth = depth > kHostMaxSlots ? kHostMaxSlots : depth;
  return depth > chunks ? chunks : depth;
}

// Calls fn(job, slot, row0, rows, index) for every chunk of the list in order
// (the schedule the call follows); stops when fn returns false.
template <typename F>
void host_for_each_chunk(const bi_host_gemm_job* jobs, int32_t n, int64_t R, int64_t depth, F fn) {
  int32_t last = -1;  // the last job with rows
  for (int32_t j = 0; j < n; ++j)
    if (jobs[j].M > 0) last = j;
  int64_t ch = 0;
  for (int32_t j = 0; j < n; ++j) {
    int64_t rows = 0;
    for (int64_t r0 = 0; r0 < jobs[j].M; r0 += rows, ++ch) {
      rows = host_next_rows(jobs[j].M - r0, R, j == last && depth >= 3);
      if (!fn(j, (int)(ch % depth), r0, rows, ch)) return;
    }
  }
}

// Every argument is checked before anything is enqueued.
bi_status host_gemm(const bi_host_gemm_job* jobs, int32_t n, int64_t N, int64_t K, const bi_pins* pins,
                    int64_t chunk_rows, void* workspace, size_t ws_bytes, cudaStream_t s) {
  int64_t R = 0, chunks = 0;
  bi_status st = host_check_rows(jobs, n, N, K, chunk_rows, &R, &chunks);
  if (st != BI_OK) return st;
  Resolved r;
  st = resolve_pins(N, K, pins, &r);
  if (st != BI_OK) return st;
  if (chunks == 0) return BI_OK;
  for (int32_t j = 0; j < n; ++j) {
    if (jobs[j].M == 0) continue;
    if (!jobs[j].X_host || !jobs[j].W || !jobs[j].Y_host) return BI_ERR_INVALID_ARG;
    if (!aligned16(jobs[j].W)) return BI_ERR_ALIGNMENT;
  }
  const uint64_t slot = host_slot_bytes(R, N, K), xoff = round256((uint64_t)R * (uint64_t)K * 2u);
  if (!workspace || ws_bytes < host_workspace_bytes(jobs, n, N, K, chunk_rows)) return BI_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BI_ERR_ALIGNMENT;
  const int64_t depth = host_depth(ws_bytes, slot, chunks);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BI_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_host_mu[dev]);
  HostCtx& c = g_host_ctx[dev];
  if (!host_ctx_init(c)) return BI_ERR_CUDA;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // everything before this call on `s` (W, the workspace's last users) comes first
  if (!ok(cudaEventRecord(c.start, s)) || !ok(cudaStreamWaitEvent(c.in, c.start, 0)) ||
      !ok(cudaStreamWaitEvent(c.out, c.start, 0)))
    return BI_ERR_CUDA;
  bi_status result = BI_OK;
  host_for_each_chunk(jobs, n, R, depth, [&](int32_t j, int i, int64_t r0, int64_t rows, int64_t ch) {
    const bi_host_gemm_job& job = jobs[j];
    char* xd = static_cast<char*>(workspace) + (uint64_t)i * slot;
    char* yd = xd + xoff;
    // the slot's previous chunk has been copied out (so also multiplied)
    if (ch >= depth && !ok(cudaStreamWaitEvent(c.in, c.copied_out[i], 0))) {
      result = BI_ERR_CUDA;
      return false;
    }
    if (!ok(cudaMemcpyAsync(xd, static_cast<const char*>(job.X_host) + (uint64_t)r0 * K * 2, (size_t)rows * K * 2,
                            cudaMemcpyHostToDevice, c.in)) ||
        !ok(cudaEventRecord(c.copied_in[i], c.in)) || !ok(cudaStreamWaitEvent(s, c.copied_in[i], 0))) {
      result = BI_ERR_CUDA;
      return false;
    }
    result = gemm_impl(xd, job.W, yd, rows, N, K, pins, s);
    if (result != BI_OK) return false;
    if (!ok(cudaEventRecord(c.multiplied[i], s)) || !ok(cudaStreamWaitEvent(c.out, c.multiplied[i], 0)) ||
        !ok(cudaMemcpyAsync(static_cast<char*>(job.Y_host) + (uint64_t)r0 * N * 2, yd, (size_t)rows * N * 2,
                            cudaMemcpyDeviceToHost, c.out)) ||
        !ok(cudaEventRecord(c.copied_out[i], c.out))) {
      result = BI_ERR_CUDA;
      return false;
    }
    return true;
  });
  // the caller's stream resumes once every copy enqueued so far has landed
  // (also after an error, so that no copy outlives the call's buffers
  // unseen by the caller's stream)
  const bool joined_in = ok(cudaEventRecord(c.end, c.in)) && ok(cudaStreamWaitEvent(s, c.end, 0));
  const bool joined_out = ok(cudaEventRecord(c.end, c.out)) && ok(cudaStreamWaitEvent(s, c.end, 0));
  if (result == BI_OK && !(joined_in && joined_out)) result = BI_ERR_CUDA;
  return result;
}

}  // namespace
}  // namespace bi

using namespace bi;

BI_API int32_t bi_abi_version(void) { return BI_PINS_ABI_VERSION; }

BI_API const char* bi_status_string(bi_status s) {
  switch (s) {
    case BI_OK: return "BI_OK";
    case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG: invalid argument";
    case BI_ERR_ALIGNMENT: return "BI_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case BI_ERR_UNSUPPORTED_SHAPE: return "BI_ERR_UNSUPPORTED_SHAPE: unsupported shape";
    case BI_ERR_ILLEGAL_PINS: return "BI_ERR_ILLEGAL_PINS: pins refused by validation";
    case BI_ERR_CUDA: return "BI_ERR_CUDA: CUDA runtime error";
    case BI_ERR_DEVICE_TIMEOUT: return "BI_ERR_DEVICE_TIMEOUT: a kernel's bounded wait ran out";
    case BI_ERR_WORKSPACE: return "BI_ERR_WORKSPACE: workspace missing or too small";
    case BI_ERR_DEBUG_BOUNDS: return "BI_ERR_DEBUG_BOUNDS: a kernel's index check failed (debug-bounds build)";
  }
  return "BI_ERR_UNKNOWN";
}

BI_API int32_t bi_debug_bounds_enabled(void) {
#ifdef BI_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

BI_API bi_status bi_debug_bounds_detail(uint64_t* detail, bi_stream_t stream) {
  if (!detail) return BI_ERR_INVALID_ARG;
  return fetch_and_clear_bounds_detail(detail, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? BI_OK
                                                                                                      : BI_ERR_CUDA;
}

BI_API bi_status bi_pins_default(int64_t N, int64_t K, bi_pins* out) { return pins_default(N, K, out); }

BI_API bi_status bi_pins_validate(int64_t N, int64_t K, const bi_pins* pins) {
  return validate(N, K, pins);
}

BI_API bi_status bi_gemm_plan_describe(int64_t M, int64_t N, int64_t K, const bi_pins* pins,
                                       int32_t sm_count, bi_gemm_plan* plan) {
  if (!plan) return BI_ERR_INVALID_ARG;
  if (M < 0) return BI_ERR_INVALID_ARG;
  bi_status st = check_nk(N, K);
  if (st != BI_OK) return st;
  Resolved r;
  st = resolve_pins(N, K, pins, &r);
  if (st != BI_OK) return st;
  return make_plan(M, N, K, r, sm_count > 0 ? sm_count : kDefaultSmCount, plan);
}

BI_API bi_status bi_gemm_bf16(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                              const bi_pins* pins, bi_stream_t stream) {
  return gemm_impl(X, W, Y, M, N, K, pins, reinterpret_cast<cudaStream_t>(stream));
}

BI_API size_t bi_gemm_bf16_workspace_bytes(int64_t M, int64_t N, int64_t K, const bi_pins* pins) {
  if (M <= 0 || check_nk(N, K) != BI_OK || M > 0x7FFFFFFFll) return 0;
  Resolved r;
  if (resolve_pins(N, K, pins, &r) != BI_OK) return 0;
  bi_gemm_plan plan;
  if (make_plan(M, N, K, r, sm_count_current(), &plan, (size_t)-1) != BI_OK) return 0;
  return plan.schedule == BI_FLAG_SCHEDULE_GLOBAL ? fold_bytes(plan) : 0;
}

BI_API bi_status bi_gemm_plan_describe_ws(int64_t M, int64_t N, int64_t K, const bi_pins* pins, int32_t sm_count,
                                          size_t workspace_bytes, bi_gemm_plan* plan) {
  if (!plan) return BI_ERR_INVALID_ARG;
  if (M < 0) return BI_ERR_INVALID_ARG;
  bi_status st = check_nk(N, K);
  if (st != BI_OK) return st;
  Resolved r;
  st = resolve_pins(N, K, pins, &r);
  if (st != BI_OK) return st;
  return make_plan(M, N, K, r, sm_count > 0 ? sm_count : kDefaultSmCount, plan, workspace_bytes);
}

BI_API bi_status bi_gemm_bf16_ws(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                                 const bi_pins* pins, void* workspace, size_t ws_bytes, bi_stream_t stream) {
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BI_ERR_ALIGNMENT;
  return gemm_impl(X, W, Y, M, N, K, pins, reinterpret_cast<cudaStream_t>(stream), Elem::BF16, nullptr, nullptr,
                   workspace, workspace ? ws_bytes : 0);
}

BI_API bi_status bi_pins_default_fp8(int64_t N, int64_t K, bi_pins* out) {
  return pins_default(N, K, out, Elem::E4M3);
}

BI_API bi_status bi_pins_validate_fp8(int64_t N, int64_t K, const bi_pins* pins) {
  return validate(N, K, pins, Elem::E4M3);
}

BI_API bi_status bi_gemm_plan_describe_fp8(int64_t M, int64_t N, int64_t K, const bi_pins* pins,
                                           int32_t sm_count, bi_gemm_plan* plan) {
  if (!plan) return BI_ERR_INVALID_ARG;
  if (M < 0) return BI_ERR_INVALID_ARG;
  bi_status st = check_nk(N, K, Elem::E4M3);
  if (st != BI_OK) return st;
  Resolved r;
  st = resolve_pins(N, K, pins, &r, Elem::E4M3);
  if (st != BI_OK) return st;
  return make_plan(M, N, K, r, sm_count > 0 ? sm_count : kDefaultSmCount, plan);
}

BI_API bi_status bi_gemm_fp8(const void* Xq, const float* sx, const void* Wq, const float* sw, void* Y,
                             int64_t M, int64_t N, int64_t K, const bi_pins* pins, bi_stream_t stream) {
  return gemm_impl(Xq, Wq, Y, M, N, K, pins, reinterpret_cast<cudaStream_t>(stream), Elem::E4M3, sx, sw);
}

BI_API bi_status bi_quantize_rows_e4m3(const void* X, void* Q, float* scale, int64_t M, int64_t K,
                                       bi_stream_t stream) {
  if (M < 0 || K < 1) return BI_ERR_INVALID_ARG;
  if (K % 16 != 0 || K > 0x7FFFFFFFll || M > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!X || !Q || !scale) return BI_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Q) || (reinterpret_cast<uintptr_t>(scale) & 3u)) return BI_ERR_ALIGNMENT;
  return launch_quantize_e4m3(X, Q, scale, M, K, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

BI_API bi_status bi_rmsnorm_quantize_e4m3(const void* X, const void* g, void* Q, float* scale, int64_t M,
                                          int64_t H, float eps, bi_stream_t stream) {
  bi_status st = check_rmsnorm_args(X, g, Q, M, H, eps);
  if (st != BI_OK) return st;
  if (H % 16 != 0 || H > kRqMaxH) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!scale) return BI_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(scale) & 3u) return BI_ERR_ALIGNMENT;
  return launch_rmsnorm_quantize_e4m3(X, g, Q, scale, M, H, eps, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

BI_API bi_status bi_rmsnorm_bf16(const void* X, const void* g, void* Y, int64_t M, int64_t H,
                                 float eps, bi_stream_t stream) {
  bi_status st = check_rmsnorm_args(X, g, Y, M, H, eps);
  if (st != BI_OK || M == 0) return st;
  return launch_rmsnorm(X, g, Y, M, H, eps, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

BI_API size_t bi_gemm_bf16_host_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const bi_host_gemm_job job = {nullptr, nullptr, nullptr, M};
  return host_workspace_bytes(&job, 1, N, K, 0);
}

BI_API bi_status bi_gemm_bf16_host(const void* X_host, const void* W, void* Y_host, int64_t M, int64_t N,
                                   int64_t K, const bi_pins* pins, void* workspace, size_t ws_bytes,
                                   bi_stream_t stream) {
  const bi_host_gemm_job job = {X_host, W, Y_host, M};
  return host_gemm(&job, 1, N, K, pins, 0, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

BI_API size_t bi_gemm_bf16_host_batch_workspace_bytes(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N,
                                                      int64_t K, int64_t chunk_rows) {
  return host_workspace_bytes(jobs, n_jobs, N, K, chunk_rows);
}

BI_API size_t bi_gemm_bf16_host_slot_bytes(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N, int64_t K,
                                           int64_t chunk_rows) {
  if (n_jobs <= 0 || !jobs || N <= 0 || K <= 0) return 0;
  int64_t R = 0, chunks = 0;
  if (!host_chunking(jobs, n_jobs, K, chunk_rows, &R, &chunks) || chunks == 0) return 0;
  return (size_t)host_slot_bytes(R, N, K);
}

BI_API bi_status bi_gemm_bf16_host_batch(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N, int64_t K,
                                         const bi_pins* pins, int64_t chunk_rows, void* workspace,
                                         size_t ws_bytes, bi_stream_t stream) {
  return host_gemm(jobs, n_jobs, N, K, pins, chunk_rows, workspace, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_gemm_bf16_host_schedule(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N, int64_t K,
                                            int64_t chunk_rows, size_t workspace_bytes, bi_host_chunk* chunks,
                                            int64_t max_chunks, int64_t* n_chunks) {
  if (!n_chunks || max_chunks < 0 || (max_chunks > 0 && !chunks)) return BI_ERR_INVALID_ARG;
  *n_chunks = 0;
  int64_t R = 0, count = 0;
  bi_status st = host_check_rows(jobs, n_jobs, N, K, chunk_rows, &R, &count);
  if (st != BI_OK || count == 0) return st;
  if (workspace_bytes < host_workspace_bytes(jobs, n_jobs, N, K, chunk_rows)) return BI_ERR_WORKSPACE;
  const int64_t depth = host_depth(workspace_bytes, host_slot_bytes(R, N, K), count);
  int64_t total = 0;
  host_for_each_chunk(jobs, n_jobs, R, depth, [&](int32_t j, int i, int64_t r0, int64_t rows, int64_t ch) {
    if (ch < max_chunks) chunks[ch] = bi_host_chunk{j, i, r0, rows};
    total = ch + 1;
    return true;
  });
  *n_chunks = total;
  return BI_OK;
}

BI_API size_t bi_rmsnorm_gemm_workspace_bytes(int64_t M, int64_t K) { return fused_workspace_bytes(M, K); }

BI_API bi_status bi_rmsnorm_gemm_bf16(const void* X, const void* g, const void* W, void* Y,
                                      int64_t M, int64_t N, int64_t K, float eps,
                                      const bi_pins* pins, void* workspace, size_t ws_bytes,
                                      bi_stream_t stream) {
  // The workspace: the RMSNorm's scratch (r, the staged rows) at its end,
  // and in front of it, when there is room, the GEMM's fold workspace (its
  // counters at offset 0 whatever M is, so that they stay zero between calls).
  const size_t base = fused_workspace_bytes(M, K);
  const bool ws_ok = workspace && ws_bytes >= base && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0;
  const size_t front = ws_ok ? ((ws_bytes - base) & ~(size_t)255) : 0;
  GemmLaunch L;
  bi_status st = plan_fused(X, g, W, Y, M, N, K, eps, pins, reinterpret_cast<cudaStream_t>(stream), &L,
                            front ? workspace : nullptr, front);
  if (st != BI_OK || L.M == 0) return st;
  if (!workspace || ws_bytes < base) return BI_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BI_ERR_ALIGNMENT;
  return launch_fused(L, static_cast<char*>(workspace) + front, fused_in_smem(L));
}

BI_API bi_status bi_residual_add_bf16(const void* a, const void* b, void* out, int64_t count,
                                      bi_stream_t stream) {
  if (count < 0) return BI_ERR_INVALID_ARG;
  if (count % 8 != 0) return BI_ERR_UNSUPPORTED_SHAPE;
  if (count == 0) return BI_OK;
  if (!a || !b || !out) return BI_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(out)) return BI_ERR_ALIGNMENT;
  return launch_residual_add(a, b, out, count, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

namespace bi {
namespace {
bi_status check_logits(const void* X, const void* out, int64_t M, int64_t V) {
  if (M < 0 || V < 1) return BI_ERR_INVALID_ARG;
  if (V % 8 != 0 || V > 0x7FFFFFFFll || M > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!X || !out) return BI_ERR_INVALID_ARG;
  if (!aligned16(X)) return BI_ERR_ALIGNMENT;
  return BI_OK;
}
}  // namespace
}  // namespace bi

BI_API bi_status bi_log_softmax_bf16(const void* X, float* Y, int64_t M, int64_t V, bi_stream_t stream) {
  bi_status st = check_logits(X, Y, M, V);
  if (st != BI_OK || M == 0) return st;
  if (!aligned16(Y)) return BI_ERR_ALIGNMENT;
  return launch_log_softmax(X, Y, M, V, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

BI_API bi_status bi_token_logprobs_bf16(const void* X, const int32_t* ids, float* out, int64_t M,
                                        int64_t V, bi_stream_t stream) {
  bi_status st = check_logits(X, out, M, V);
  if (st != BI_OK || M == 0) return st;
  if (!ids) return BI_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ids) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u))
    return BI_ERR_ALIGNMENT;
  return launch_token_logprobs(X, ids, out, M, V, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

namespace {

bi_status attn_geometry(int64_t B, int64_t Hq, int64_t Hkv, int64_t max_seq_len, int64_t* split,
                        int64_t* n_split, int64_t* gp) {
  if (B < 0 || Hq < 1 || Hkv < 1 || max_seq_len < 0 || *split < 0) return BI_ERR_INVALID_ARG;
  if (*split == 0) *split = BI_ATTN_DEFAULT_SPLIT;
  if (Hq % Hkv != 0 || Hq / Hkv > 16 || *split % 64 != 0 || *split > BI_ATTN_MAX_SPLIT || B > 65535 ||
      Hkv > 65535 || Hq > (int64_t)1 << 20 || max_seq_len > ((int64_t)1 << 40))
    return BI_ERR_UNSUPPORTED_SHAPE;
  *n_split = std::max<int64_t>(1, (max_seq_len + *split - 1) / *split);
  // item entries pack (request, split) into 16 bits each; tickets are 32-bit
  if (*n_split > 65535 || B * *n_split * Hkv >= ((int64_t)1 << 31)) return BI_ERR_UNSUPPORTED_SHAPE;
  *gp = Hq / Hkv <= 8 ? 8 : 16;
  return BI_OK;
}

int32_t log2_pow2(int64_t v) {
  int32_t s = 0;
  while (((int64_t)1 << s) < v) ++s;
  return s;
}

// Workspace: 256 bytes of control words (ticket counter, item count), the
// item list (one uint32 per (request, split), padded to 256 bytes), then the
// split records (B * Hkv * n_split of (128 + 2) * GP floats).
int64_t attn_list_bytes(int64_t B, int64_t n_split) { return (B * n_split * 4 + 255) / 256 * 256; }

int64_t attn_ws_bytes(int64_t B, int64_t Hkv, int64_t n_split, int64_t gp) {
  return 256 + attn_list_bytes(B, n_split) + B * Hkv * n_split * (BI_ATTN_HEAD_DIM + 2) * gp * 4;
}

// A paged cache [num_pages, page_size, Hkv, 128] seen as [rows][2 Hkv][64]:
// position, 64-value half of a head, value.  A box is {64 values, the two
// halves of one head, box_rows positions}, landing as 2 box_rows rows of
// 128 bytes (position-major).
bool encode_cache(CUtensorMap* map, const void* ptr, int64_t rows, int64_t Hkv, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)(Hkv * 2), (cuuint64_t)rows};
  cuuint64_t strides[2] = {128, (cuuint64_t)(Hkv * BI_ATTN_HEAD_DIM * 2)};
  cuuint32_t box[3] = {64, 2, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

BI_API bi_status bi_decode_attention_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t max_seq_len,
                                                     int64_t split_size, size_t* bytes) {
  if (!bytes) return BI_ERR_INVALID_ARG;
  int64_t n_split = 0, gp = 0;
  bi_status st = attn_geometry(B, Hq, Hkv, max_seq_len, &split_size, &n_split, &gp);
  if (st != BI_OK) return st;
  *bytes = (size_t)attn_ws_bytes(B, Hkv, n_split, gp);
  return BI_OK;
}

BI_API bi_status bi_decode_attention_bf16(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                                          void* out, int64_t B, int64_t Hq, int64_t Hkv, int64_t D,
                                          int64_t num_pages, int64_t page_size, int64_t max_seq_len,
                                          int64_t split_size, float scale, void* ws, size_t ws_bytes,
                                          bi_stream_t stream) {
  int64_t n_split = 0, gp = 0;
  bi_status st = attn_geometry(B, Hq, Hkv, max_seq_len, &split_size, &n_split, &gp);
  if (st != BI_OK) return st;
  if (num_pages < 1 || page_size < 1 || bt_stride < 0 || !std::isfinite(scale)) return BI_ERR_INVALID_ARG;
  if (D != BI_ATTN_HEAD_DIM || page_size < 8 || (page_size & (page_size - 1)) != 0 ||
      num_pages > 0x7FFFFFFFll / page_size)
    return BI_ERR_UNSUPPORTED_SHAPE;
  if (bt_stride < (max_seq_len + page_size - 1) / page_size) return BI_ERR_INVALID_ARG;
  if (B == 0) return BI_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !ws) return BI_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return BI_ERR_ALIGNMENT;
  if (ws_bytes < (size_t)attn_ws_bytes(B, Hkv, n_split, gp)) return BI_ERR_WORKSPACE;
  AttnLaunch A = {};
  const int box_rows = (int)std::min<int64_t>(page_size, 32);  // one 32-position tile at most
  if (!encode_cache(&A.tmK, k_cache, num_pages * page_size, Hkv, box_rows) ||
      !encode_cache(&A.tmV, v_cache, num_pages * page_size, Hkv, box_rows))
    return BI_ERR_CUDA;
  A.p.q = q;
  A.p.block_table = block_table;
  A.p.seq_lens = seq_lens;
  A.p.ctl = static_cast<uint32_t*>(ws);
  A.p.items = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + 256);
  A.p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + 256 + attn_list_bytes(B, n_split));
  A.p.bt_stride = bt_stride;
  A.p.num_pages = num_pages;
  A.p.max_len = max_seq_len;
  A.p.Hq = (int32_t)Hq;
  A.p.Hkv = (int32_t)Hkv;
  A.p.G = (int32_t)(Hq / Hkv);
  A.p.page_size = (int32_t)page_size;
  A.p.box_rows = box_rows;
  A.p.page_shift = log2_pow2(page_size);
  A.p.box_shift = log2_pow2(box_rows);
  A.p.nreq = (int32_t)B;
  A.p.split_size = (int32_t)split_size;
  A.p.n_split = (int32_t)n_split;
  A.p.qk_log2 = (float)((double)scale * 1.4426950408889634);  // scale * log2(e)
  A.p.status = device_status_word();
  if (!A.p.status) return BI_ERR_CUDA;
  A.out = out;
  A.B = B;
  A.grid = sm_count_current();
  A.stream = reinterpret_cast<cudaStream_t>(stream);
  return launch_decode_attention(A) == cudaSuccess ? BI_OK : BI_ERR_CUDA;
}

BI_API bi_status bi_silu_mul_bf16(const void* gu, void* out, int64_t M, int64_t I,
                                  bi_stream_t stream) {
  if (M < 0 || I < 1) return BI_ERR_INVALID_ARG;
  if (I % 8 != 0) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!gu || !out) return BI_ERR_INVALID_ARG;
  if (!aligned16(gu) || !aligned16(out)) return BI_ERR_ALIGNMENT;
  return launch_silu_mul(gu, out, M, I, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

BI_API bi_status bi_attention_ctx1_bf16(const void* qkv, void* out, int64_t M, int64_t nq,
                                        int64_t nkv, int64_t D, bi_stream_t stream) {
  if (M < 0 || nq < 1 || nkv < 1 || D < 1) return BI_ERR_INVALID_ARG;
  if (nq % nkv != 0 || D % 8 != 0) return BI_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return BI_OK;
  if (!qkv || !out) return BI_ERR_INVALID_ARG;
  if (!aligned16(qkv) || !aligned16(out)) return BI_ERR_ALIGNMENT;
  return launch_attention_ctx1(qkv, out, M, nq, nkv, D, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? BI_OK
             : BI_ERR_CUDA;
}

BI_API bi_status bi_last_device_status(bi_stream_t stream) {
  int v = 0;
  if (fetch_and_clear_stall(&v, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BI_ERR_CUDA;
  // the word holds the first code a kernel recorded since the last read
  return v == 0 ? BI_OK : (bi_status)v;
}
