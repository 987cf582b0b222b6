// gemm.cu -- FP8 e4m3 block-scaled GEMM for sm_103a: dense NT, contiguous-grouped and
// masked-grouped MoE forms, one persistent warp-specialised kernel template.
//
// What is computed ("DeepGEMM FP8 walk-through" sec. 2.2-2.3, "DeepGEMM explainer"
// sec. 3.1-3.3): D = bf16( sum_kb P_kb * sA[kb][m] * sB[n/128][kb] ), P_kb the e4m3 x e4m3
// product of one 128-wide K block, accumulated in FP32.  The scales are applied inside the
// GEMM pipeline, not by a separate dequantisation pass.
//
// GB300 design (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0        TMA producer: A tile (128 x 128 B) and B tile (BN x 128 B) of each K block
//                 into one stage of a STAGES-deep shared-memory ring, signalled through a
//                 full/empty mbarrier pair per stage (two TMA instructions per K block).
//   warp 1        allocates TMEM; one lane issues 4 tcgen05.mma kind::f8f6f4 (K = 32 each)
//                 per K block into a FRESH TMEM partial (the first MMA does not accumulate),
//                 in a ring of TMEM buffers (2 at BN = 256, up to 8 for narrow tiles) so the
//                 MMA of later K blocks overlaps the promotion of earlier ones.
//   warps 2.. /4..  promotion + epilogue: tcgen05.ld the partial (64 columns per load), then
//                 acc = fma(P, sa*sb, acc) in FP32 registers with packed FP32 FMAs (one TMEM
//                 lane = one output row per thread).  sa (one per row and K block) is read
//                 from global memory a few K blocks ahead; sb (one per 128 columns and K
//                 block) is held in a register per lane and broadcast by shuffle.  After the
//                 last K block: BF16, staged in shared memory, stored with TMA (64-byte
//                 swizzled 32 x 32 boxes).  Rows past a masked expert's count are never
//                 written.  Narrow tiles (BN = 64) split the K blocks between two warpgroups.
// Epilogue-scaled variant (EPI; per-tensor / per-token / per-channel scales, "DeepGEMM FP8
// walk-through" sec. 2.2, the fused epilogue of the Triton listing on "Production FP8 GEMM
// alignment and Tensor Core peak tuning"): the MMAs of all K blocks of a tile accumulate in
// place in one TMEM buffer (2 at BN = 256: the epilogue of one tile overlaps the MMAs of the
// next), each K block's commit frees its stage, and the epilogue reads the accumulator once and
// multiplies it by sa[m] * sb[n] before the BF16 store.
// Backward forms (e5m2 gradients, "E4M3 vs E5M2" on the Production FP8 GEMM page): the operand
// formats are a run-time field of the MMA instruction descriptor (A in e5m2 for the data
// gradient), and the K-grouped mode computes one weight-gradient matrix per expert over that
// expert's token range, with a B scale per column and K block applied in the promotion.
// Stream-K tail: when the tiles do not fill whole rounds of the grid, the last round's K blocks
// are split over all SMs and the partial sums are added by the CTA holding each tile's start.
// Every wait is bounded: a wait that runs past its cycle budget records FP8G_ERR_TIMEOUT in
// the status word, raises a shared abort flag, and every role returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8g {
namespace {

// kDenseSmallM: dense with M <= 64 (decode shapes), BN = 64 only: loads 64 A rows per stage.
// kKGrouped: the weight gradient of a grouped layer -- one output matrix per expert, the
// contraction running over that expert's token range (offsets in the group table), both
// operands with one scale per row and 128-token block.
// kSwapAB (opt-in, FP8G_SWAP_AB=1): dense with M <= 64 computed as D^T = B A^T: the weight rows
// take the MMA's M = 128 (a tile is a 128-row weight slab) and the tokens its N = 64, so each
// tcgen05.mma covers twice the weight bytes of a 64-wide tile.  The tensor maps are swapped on
// the host ("A" is the weight, "B" the activations); the promotion takes one weight-block scale
// per tile and K block and one activation scale per column; the output is stored transposed.
// The few tiles (N / 128) have their K blocks split over all SMs by the stream-K tail.
enum Mode : int { kDense = 0, kContiguous = 1, kMasked = 2, kDenseSmallM = 3, kKGrouped = 4, kSwapAB = 5 };

constexpr int BM = 128;  // rows per tile = TMEM lanes
constexpr int BK = 128;  // K per stage = the scaling block
constexpr int kBandM = 16;  // m-blocks per raster band of CTA pairs (L2 reuse of B across a band)

// PAIR: a cluster of two CTAs computes 256 x BN tiles with tcgen05.mma.cta_group::2; each CTA
// loads its 128 A rows and half of the B tile (BN / 2 rows), so a stage is 32 KB and six fit.
// KG: the K-grouped weight gradient, whose tiles are short (one expert's tokens): three stages
// (its operands come mostly from L2) make room for a staging box per 32 columns in every store
// warp, so a tile's boxes are stored without waiting on one another, and for each epilogue
// warp's 512 bytes of per-column B scales.
template <int BN, bool SMALL = false, bool PAIR = false, bool KG = false, bool SWAP = false>
struct Cfg {
  // columns per epilogue warp.  192-wide tiles and 256 x 128 pair tiles: 64, 160-wide tiles: 32,
  // so that each warp reads its whole partial with one load and frees the TMEM buffer before any
  // FMA (a 128-column warp holds 128 accumulators and can load only half its partial at a time, so
  // the FMAs of the first half sit between the buffer's completion and its release).
  // Swapped tiles (64 token columns): 32, eight warps (per thread 32 accumulators, 32 loaded values
  // and two prefetched sets of 32 column scales, with the registers of the rebalance below).
  static constexpr int kEpiCols =
      (BN == 160 || SWAP) ? 32 : (((PAIR && BN == 128) || BN == 192) ? 64 : (BN >= 128 ? 128 : BN));
  static constexpr int kColGroups = BN / kEpiCols;       // warpgroups covering the tile's columns
  // Narrow tiles (few, long K loops: small-M shapes) split the K blocks between two sets of
  // promotion warps (even / odd K blocks), whose FP32 partial sums are added at the tile end.
  static constexpr int kKSplit = ((BN == 64 || BN == 48) && !SWAP) ? 2 : 1;
  static constexpr int kEpiGroups = kColGroups * kKSplit;  // warpgroups of epilogue warps
  static constexpr int kEpiWarps = 4 * kEpiGroups;
  static constexpr int kStoreWarps = 4 * kColGroups;     // warps that write D
  // MMA issuing threads (lane 0 of warps 1 .. kMmaWarps), taking the pipeline stages in turn.
  // One thread pays ~60 cycles per tcgen05.mma plus ~170 per mbarrier round trip, which caps
  // the narrow small-M tiles (whose MMAs are short); there three issuers share the stream (one:
  // 22.6 us for 64 x 7168 x 7168, two: 17.4, three: 16.8).  Wider tiles keep one: their MMAs
  // are long enough, and measured slower with two.
  // 256 x 128 pair tiles: four MMAs of ~64 cycles per K block for the pair, so two lone issuers;
  // 160-wide tiles: four MMAs of ~81 cycles per K block, also two.
  static constexpr int kMmaWarps = SMALL ? 3 : (((PAIR && BN == 128) || BN == 160) ? 2 : 1);
  // BN = 256, 192 and 160: a full first warpgroup (producer / MMA / idle) then the epilogue
  // warpgroups, so that setmaxnreg can move registers to the epilogue.  BN = 256: the launch gives
  // 384 x 168 = 64512, rebalanced to 128 x 40 + 256 x 232 = 64512.  BN = 192: 512 x 128 = 65536,
  // rebalanced to 128 x 32 + 384 x 160 = 65536 (64 accumulators and 64 loaded values a thread).
  // BN = 160: 768 x 80 = 61440, rebalanced to 128 x 40 + 640 x 88 = 61440 (32 accumulators and 32
  // loaded values).  Swapped tiles: 384 x 168, rebalanced as at BN = 256.  Otherwise: producer and
  // MMA warps, then the epilogue warpgroups (any four consecutive warps cover the four TMEM lane
  // quarters).
  static constexpr bool kRebalance = BN == 256 || BN == 192 || BN == 160 || SWAP;
  static constexpr int kEpiWarp0 = kRebalance ? 4 : 1 + kMmaWarps;
  static constexpr int kThreads = 32 * kEpiWarp0 + 32 * kEpiWarps;
  static constexpr uint32_t kRegsLow = BN == 192 ? 32 : 40;
  static constexpr uint32_t kRegsHigh = (BN == 256 || SWAP) ? 232 : (BN == 192 ? 160 : 88);
  // A rows loaded per stage: the MMA always reads 128 rows, and with SMALL the upper 64 are
  // whatever follows in shared memory (those rows of D are computed but never stored).
  static constexpr int kARows = SMALL ? 64 : BM;
  // K blocks per pipeline stage.  One TMA box then covers kKPS consecutive 128-byte pieces of
  // every row (a kKPS * 128-byte run in global memory): streaming weights from HBM in 128-byte
  // pieces of rows 7 KB apart reaches about half the bandwidth of 256-byte runs.
  static constexpr int kKPS = (SMALL || SWAP) ? 2 : 1;
  // (swapped tiles: 32 KB of weights and 16 KB of activations per stage)
  // (a multiple of the lone issuers' count: see the assertion below)
  static constexpr int kStages =
      SMALL ? 6 : (SWAP ? 4 : (PAIR ? (BN == 256 ? 5 : 8) : (KG ? 3 : (BN >= 192 ? 4 : (BN == 160 ? 4 : 6)))));
  // TMEM partial buffers: as many as fit the 512 columns, so the MMA can run ahead of the
  // promotion by several K blocks (2 at BN = 256, 3 at 160, 4 at 128, 8 at 64).
  static constexpr int kTmemBufs = 512 / BN > 8 ? 8 : 512 / BN;
  // TMEM columns between buffers: BN, but 64 for the 48-wide tiles (each buffer then starts on a
  // 64-column boundary, as in the 64-wide tiles)
  static constexpr uint32_t kTmemStride = BN == 48 ? 64u : static_cast<uint32_t>(BN);
  static_assert(kTmemBufs * kTmemStride <= 512, "TMEM buffers");
  // Small-M tiles synchronise the MMA and the promotion once per stage, not once per K block:
  // a stage's kKPS partials go to one TMEM slot of kKPS buffers, completed by one commit, and the
  // slot is written again once every promotion warp (both K parts) has read its K block of it.
  // The lone issuers' barrier round trips (~100-200 cycles each) otherwise set the pace of these
  // short MMAs.
  static constexpr bool kStageSync = SMALL;
  static constexpr uint32_t kSlotCols = kStageSync ? static_cast<uint32_t>(kKPS) * kTmemStride : kTmemStride;
  static constexpr uint32_t kTmemSlots = kStageSync ? 512u / kSlotCols : static_cast<uint32_t>(kTmemBufs);
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kABytes = kARows * BK;       // one K block of A
  static constexpr int kBRows = PAIR ? BN / 2 : BN;      // B rows this CTA loads
  static constexpr uint32_t kBBytes = kBRows * BK;       // one K block of B
  static constexpr uint32_t kStageABytes = kKPS * kABytes;
  static constexpr uint32_t kStageBBytes = kKPS * kBBytes;
  static constexpr uint32_t kOutBytes = 32 * 32 * 2;  // one 32 x 32 bf16 box
  // staging boxes per store warp (swapped tiles store with plain transposed stores: none)
  static constexpr int kOutBoxes = SWAP ? 0 : (KG ? kEpiCols / 32 : 1);
  static constexpr uint32_t kOutWarpBytes = kOutBoxes * kOutBytes;
  // K-grouped: the scales of each stage's K block, staged next to its operands by the producer --
  // the tile's 128 A-row scales (a 512-byte TMA box) and its BN per-column B scales (a TMA box).
  // (The block forms read their two scales per K block from global memory, well ahead of use.)
  static constexpr uint32_t kSAKB = BM * 4;
  static constexpr uint32_t kSBKB = BN * 4;
  static constexpr uint32_t kScaleStage = KG ? kSAKB + kSBKB : 0u;
  // K-grouped: each epilogue warp copies its 128 columns' B scales out of the stage (512 bytes)
  static constexpr uint32_t kSbvBytes = KG ? 512u * kEpiWarps : 0u;
  static constexpr int kXRows = SMALL ? 64 : BM;
  static constexpr uint32_t kXBytes = kKSplit > 1 ? kXRows * BN * 4 : 0;  // K-split exchange
  // shared-memory carve-up (offsets from a 1024-aligned base)
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = kOffA + kStages * kStageABytes;
  static constexpr uint32_t kOffOut = kOffB + kStages * kStageBBytes;
  static constexpr uint32_t kOffScale = kOffOut + kStoreWarps * kOutWarpBytes;
  static constexpr uint32_t kOffSbv = kOffScale + kStages * kScaleStage;
  static constexpr uint32_t kOffX = kOffSbv + kSbvBytes;
  static constexpr uint32_t kOffBar = kOffX + kXBytes;
  static constexpr uint32_t kNumBars = 3 * kStages + 2 * kTmemBufs + 5;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffTable = kOffMisc + 16;
  static_assert(kOffA % 1024 == 0 && kOffB % 1024 == 0 && kOffOut % 1024 == 0, "alignment");
  static_assert(kOffScale % 128 == 0 && kScaleStage % 128 == 0 && kOffSbv % 16 == 0, "scale staging alignment");
  static_assert(BN == 48 || BN == 64 || BN == 128 || BN == 160 || BN == 192 || BN == 256, "BN");
  static_assert(BN != 48 || SMALL, "48-wide tiles: the small-M variant");
  static_assert((BN != 192 && BN != 160) || (!SMALL && !PAIR && !KG),
                "160- and 192-wide tiles: single-CTA block-scaled forms");
  static_assert(!SMALL || BN == 64 || BN == 48, "small-M tiles are 64 or 48 wide");
  static_assert(!SWAP || (BN == 64 && !SMALL && !PAIR && !KG), "swapped tiles: 64 token columns, single CTA");
  static_assert(!PAIR || ((BN == 256 || BN == 128) && !SMALL), "CTA pairs use 128- or 256-wide tiles");
  static_assert(kEpiWarp0 > kMmaWarps, "producer and MMA warps precede the epilogue");
  // Lone issuers wait for a stage's operands by the parity of its full barrier's phase, which is
  // only sound if the stage's previous fill (kStages stages earlier) has landed.  Copies may land
  // out of order, so an issuer knows that only of the stages it consumed itself: each stage slot
  // must always go to the same issuer.
  static_assert(kMmaWarps == 1 || kStages % kMmaWarps == 0, "lone issuers: one issuer per stage slot");
  static_assert(!kStageSync || (kKSplit == 2 && kKPS == 2 && kMmaWarps >= 2),
                "stage-synchronised tiles: K part j reads K block j of every stage, lone issuers");
};

// The configuration of a kernel instantiation.
template <int BN, int MODE, bool PAIR>
using CfgOf = Cfg<BN, MODE == kDenseSmallM, PAIR, MODE == kKGrouped, MODE == kSwapAB>;

struct GemmArgs {
  int32_t rows;      // rows of A / D (M, M_total or E*cap; swapped: the weight rows N)
  int32_t N, KB, NBs, E, cap;
  int32_t num_m;     // m-blocks (dense / contiguous)
  int32_t num_n;     // n-blocks of BN
  int32_t num_tiles; // dense / contiguous tile count
  int32_t band_m;    // m-blocks per raster band (dense / contiguous / K-grouped; see band_rows)
  const float* sA;   // A-row scales [KB][ld_sa]
  int64_t ld_sa;
  const float* sB;
  __nv_bfloat16* D;
  int64_t ldd;
  const int32_t* groups;  // contiguous: offsets [E+1]; masked: counts [E]
  unsigned int* status;
  long long budget;
  // epilogue scaling: sA holds one scale per row of A (sa_step 1) or one for all rows (0); sB one
  // per column of each expert, [E][N] (sb_step 1), or one per expert, [E] (0)
  int32_t sa_step, sb_step;
  // operand formats in the MMA instruction descriptor (A bits 7-9, B bits 10-12; 0 = e4m3, 1 = e5m2)
  uint32_t idesc_fmt;
  int64_t ld_sb;  // kKGrouped: B scales [K blocks][ld_sb], one per row of B

  // stream-K tail (see make_work): on/off, its minimum K blocks per CTA, and the workspace of
  // FP32 partial tiles (one slot per CTA) with one ready flag per CTA (zeroed before the launch)
  int32_t sk;
  int32_t sk_min_units;
  int32_t sk_min_gain;  // split only when it saves at least this many K blocks per CTA
  float4* ws_part;
  uint32_t* ws_flag;
  // cluster K split (see make_work), 0 or 1 when off: each cluster of ck CTAs computes one tile,
  // its ranks taking consecutive K ranges; rank 0 adds the others' partials (workspace slots)
  int32_t ck;

  // Test hook, -1 normally: the producer never fills its stage number `test_skip_stage` (counted
  // over the CTA's stages), so the MMA issuer's bounded wait for it runs out and the abort path
  // runs (FP8G_ERR_TIMEOUT; every role leaves, in-flight copies and MMAs are awaited, TMEM freed).
  int32_t test_skip_stage;
};

struct Tile {
  int32_t a_row;  // first row of A (and of the A scales)
  int32_t n0;     // first column
  int32_t g;      // expert
  int32_t rows;   // rows of the tile that may be stored (masked tail), else BM
  int32_t d_row;  // first row of D (a_row, except kKGrouped: expert * M + a_row)
  int32_t kb_first, kb_count;  // the tile's K blocks (0 and KB, except kKGrouped: its expert's tokens)
};

// The work of one CTA, as pieces (tile, K blocks kb0 .. kb1 - 1).  Whole tiles c, c + G, ...
// come first.  With the stream-K tail on, only the whole rounds of tiles are dealt that way; the
// K blocks of the R < G tiles left over are then split evenly over the G CTAs (CTA c takes units
// [c*u, (c+1)*u) of the tail's R*KB, u >= sk_min_units), so the last round no longer leaves most
// SMs idle.  A tile split between CTAs is finished by the CTA holding its first K blocks (it
// reaches them at the end of its share, when the others have written their partial sums): it
// adds the partials of CTAs c_lo .. c_hi and stores.  The others (kContrib) write their FP32
// partial to their workspace slot and raise their flag.  Each CTA has at most one piece of each
// of the two kinds.
enum PieceKind : int32_t { kWhole = 0, kFinish = 1, kContrib = 2 };
struct Piece {
  int32_t t, kb0, kb1, kind, c_lo, c_hi;
};
struct Work {
  int32_t G, KB, c;
  int32_t t, t_end;           // whole tiles t, t + G, ... below t_end
  int32_t tail0, u;           // first tail tile, tail K blocks per CTA
  int32_t unit, unit_end;     // this CTA's tail units
};
// Cluster K split (ck > 1; dense single-CTA tiles, one tile per cluster, ck dividing KB): the
// stream-K tail with no whole tiles and u = KB / ck, so that CTA c is rank c % ck of cluster c / ck
// and takes K blocks [(c % ck) u, (c % ck + 1) u) of tile c / ck.  Rank 0 finishes the tile with the
// partials of ranks 1 .. ck-1 (CTAs c+1 .. c+ck-1), which signal it through its shared memory: no
// flags to clear, and the cluster launch makes the ranks resident together.
__device__ __forceinline__ Work make_work(int32_t num_tiles, int32_t G, int32_t c, int32_t KB, bool sk,
                                          int32_t min_units, int32_t min_gain, int32_t ck = 0) {
  Work w;
  w.G = G;
  w.KB = KB;
  w.c = c;
  w.t = c;
  if (ck > 1) {
    w.t = w.t_end = w.tail0 = 0;
    w.u = KB / ck;
    const int64_t U = static_cast<int64_t>(num_tiles) * KB, s0 = static_cast<int64_t>(c) * w.u;
    w.unit = static_cast<int32_t>(s0 < U ? s0 : U);
    w.unit_end = static_cast<int32_t>(s0 + w.u < U ? s0 + w.u : U);
    return w;
  }
  if (!sk) {
    w.t_end = num_tiles;
    w.tail0 = num_tiles;
    w.u = 1;
    w.unit = w.unit_end = 0;
    return w;
  }
  w.tail0 = (num_tiles / G) * G;
  w.t_end = w.tail0;
  const int64_t U = static_cast<int64_t>(num_tiles - w.tail0) * KB;
  int64_t u = (U + G - 1) / G;
  const int64_t umin = min_units < KB ? min_units : KB;
  if (u < umin) u = umin;
  if (KB - u < min_gain) {  // the split would not pay for its partial-sum traffic: whole tiles
    w.t_end = num_tiles;
    w.tail0 = num_tiles;
    w.u = 1;
    w.unit = w.unit_end = 0;
    return w;
  }
  w.u = static_cast<int32_t>(u);
  const int64_t s0 = static_cast<int64_t>(c) * u;
  w.unit = static_cast<int32_t>(s0 < U ? s0 : U);
  w.unit_end = static_cast<int32_t>(s0 + u < U ? s0 + u : U);
  return w;
}
__device__ __forceinline__ bool next_piece(Work& w, Piece& p) {
  if (w.t < w.t_end) {
    p.t = w.t;
    p.kb0 = 0;
    p.kb1 = w.KB;
    p.kind = kWhole;
    p.c_lo = 0;
    p.c_hi = -1;
    w.t += w.G;
    return true;
  }
  if (w.unit < w.unit_end) {
    const int32_t r = w.unit / w.KB, kb0 = w.unit - r * w.KB;
    const int32_t take = min(w.KB - kb0, w.unit_end - w.unit);
    p.t = w.tail0 + r;
    p.kb0 = kb0;
    p.kb1 = kb0 + take;
    if (kb0 == 0 && p.kb1 == w.KB) {
      p.kind = kWhole;
      p.c_lo = 0;
      p.c_hi = -1;
    } else if (kb0 == 0) {  // the other units of tile r belong to the following CTAs
      p.kind = kFinish;
      p.c_lo = (r * w.KB + p.kb1) / w.u;
      p.c_hi = (r * w.KB + w.KB - 1) / w.u;
    } else {
      p.kind = kContrib;
      p.c_lo = p.c_hi = w.c;
    }
    w.unit += take;
    return true;
  }
  return false;
}

// Tile index -> tile.  Returns false when the tile has no rows to compute.
template <int BN, int MODE>
__device__ __forceinline__ bool get_tile(const GemmArgs& a, const int32_t* table, int32_t t,
                                         Tile& ti) {
  ti.kb_first = 0;
  ti.kb_count = a.KB;
  if (MODE == kKGrouped) {
    // expert e = t / (m-blocks x n-blocks), then the dense banded raster within the expert
    const int32_t per_e = a.num_m * a.num_n;
    const int32_t e = t / per_e, r = t - e * per_e;
    const int32_t band_tiles = a.band_m * a.num_n;
    const int32_t band = r / band_tiles, rr = r - band * band_tiles;
    const int32_t m_first = band * a.band_m;
    const int32_t gm = min(a.band_m, a.num_m - m_first);
    const int32_t mb = m_first + rr % gm, nb = rr / gm;
    ti.g = e;
    ti.a_row = mb * BM;
    ti.n0 = nb * BN;
    ti.rows = min(BM, a.rows - ti.a_row);
    ti.d_row = e * a.rows + ti.a_row;
    ti.kb_first = table[e] / BK;
    ti.kb_count = (table[e + 1] - table[e]) / BK;  // 0 for an expert without tokens: zeros
    return true;
  }
  if (MODE == kMasked) {
    // table[e] = sum of m-blocks of experts < e; an expert's tiles are (nb, mb), mb fastest
    int lo = 0, hi = a.E;  // find e with table[e]*num_n <= t < table[e+1]*num_n
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<int64_t>(table[mid]) * a.num_n <= t) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int32_t mbs = table[e + 1] - table[e];
    if (mbs <= 0) return false;
    const int32_t local = t - table[e] * a.num_n;
    const int32_t mb = local % mbs, nb = local / mbs;
    int32_t cnt = __ldg(a.groups + e);
    cnt = min(max(cnt, 0), a.cap);
    ti.g = e;
    ti.a_row = e * a.cap + mb * BM;
    ti.d_row = ti.a_row;
    ti.n0 = nb * BN;
    ti.rows = min(BM, cnt - mb * BM);
    return ti.rows > 0;
  } else {
    const int32_t band_tiles = a.band_m * a.num_n;
    const int32_t band = t / band_tiles, r = t - band * band_tiles;
    const int32_t m_first = band * a.band_m;
    const int32_t gm = min(a.band_m, a.num_m - m_first);
    const int32_t mb = m_first + r % gm, nb = r / gm;
    ti.a_row = mb * BM;
    ti.d_row = ti.a_row;
    ti.n0 = nb * BN;
    ti.rows = min(BM, a.rows - ti.a_row);  // rows past the matrix edge are not stored
    ti.g = 0;
    if (MODE == kContiguous) {
      // expert e with offsets[e] <= row < offsets[e+1]: first index with offsets[i] > row, minus 1
      int lo = 0, hi = a.E + 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (table[mid] > ti.a_row) hi = mid; else lo = mid + 1;
      }
      const int e = lo - 1;
      if (e < 0 || e >= a.E) return false;
      ti.g = e;
    }
    return true;
  }
}

// CTA-pair tile index -> this CTA's half (rank 0: the first 128 rows of the 256-row tile).
// Every pair tile is computed by both CTAs; a half whose rows are all outside the matrix or
// group has rows <= 0 and stores nothing.
template <int BN, int MODE>
__device__ __forceinline__ void get_pair_tile(const GemmArgs& a, const int32_t* table, const int32_t* ptab,
                                              int32_t t, uint32_t rank, Tile& ti) {
  ti.kb_first = 0;
  ti.kb_count = a.KB;
  if (MODE == kDense) {
    constexpr int kBand = kBandM / 2;  // pairs per raster band
    const int32_t num_mp = (a.num_m + 1) >> 1;
    const int32_t band_tiles = kBand * a.num_n;
    const int32_t band = t / band_tiles, r = t - band * band_tiles;
    const int32_t p_first = band * kBand;
    const int32_t gm = min(kBand, num_mp - p_first);
    const int32_t mp = p_first + r % gm, nb = r / gm;
    ti.a_row = (2 * mp + static_cast<int32_t>(rank)) * BM;
    ti.d_row = ti.a_row;
    ti.n0 = nb * BN;
    ti.rows = min(BM, a.rows - ti.a_row);
    ti.g = 0;
    return;
  }
  // grouped: ptab[e] = pair tiles (per column block) of experts < e; pairs m-block fastest
  int lo = 0, hi = a.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(ptab[mid]) * a.num_n <= t) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int32_t pairs = ptab[e + 1] - ptab[e];
  const int32_t local = t - ptab[e] * a.num_n;
  const int32_t pr = local % pairs, nb = local / pairs;
  const int32_t mb = 2 * pr + static_cast<int32_t>(rank);  // m-block of this CTA within the expert
  ti.g = e;
  ti.n0 = nb * BN;
  if (MODE == kContiguous) {
    const int32_t first = table[e], end = table[e + 1];
    ti.a_row = first + mb * BM;
    ti.rows = ti.a_row < end ? BM : 0;
  } else {
    int32_t cnt = __ldg(a.groups + e);
    cnt = min(max(cnt, 0), a.cap);
    ti.a_row = e * a.cap + mb * BM;
    ti.rows = min(BM, cnt - mb * BM);
  }
  ti.d_row = ti.a_row;
}

// One TMEM load of 32 or 64 columns with its wait (tcgen05.ld 32x32b.x32 / .x64).
__device__ __forceinline__ void tmem_ld_sync(uint32_t taddr, float (&v)[32]) { tmem_ld32_sync(taddr, v); }
__device__ __forceinline__ void tmem_ld_sync(uint32_t taddr, float (&v)[64]) { tmem_ld64_sync(taddr, v); }
__device__ __forceinline__ void tmem_ld_sync(uint32_t taddr, float (&v)[48]) { tmem_ld48_sync(taddr, v); }

// Bounded wait on an mbarrier phase.  On timeout: flag the CTA, record the status.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const GemmArgs& a,
                                             volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > a.budget) {
      *abort_flag = 1;
      record_status(a.status, FP8G_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Wait for a phase that an earlier mbar_test_wait may already have seen complete (`seen`).  A
// lone issuing thread pays the full round trip of every mbarrier test (~170 cycles, complete or
// not), so the producer and MMA loops start the test for their next wait before issuing the
// current copies / MMAs, and consume the result here.  A phase seen complete stays complete:
// the barrier's next phase needs this thread's own work first.
__device__ __forceinline__ bool wait_seen(bool seen, uint32_t bar, uint32_t parity, const GemmArgs& a,
                                          volatile int* abort_flag) {
  return seen || wait_bounded(bar, parity, a, abort_flag);
}

// Bounded wait for another CTA's flag (stream-K partial written).  On timeout: flag this CTA,
// record the status.
__device__ __forceinline__ bool wait_flag(const uint32_t* f, const GemmArgs& a, volatile int* abort_flag) {
  if (ld_acquire_gpu(f) != 0u) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(f) == 0u) {
    if (*abort_flag) return false;
    if (clock64() - t0 > a.budget) {
      *abort_flag = 1;
      record_status(a.status, FP8G_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

template <int BN, int MODE, bool PAIR = false, bool EPI = false>
__global__ void __launch_bounds__(CfgOf<BN, MODE, PAIR>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmSA,
                    const __grid_constant__ CUtensorMap tmSB, const GemmArgs a) {
  using C = CfgOf<BN, MODE, PAIR>;
  static_assert(!EPI || (C::kKSplit == 1 && C::kMmaWarps == 1 && !PAIR),
                "epilogue scaling: one K part, one issuer, single-CTA tiles");
  static_assert(MODE != kKGrouped || (!EPI && !PAIR && C::kMmaWarps == 1),
                "K-grouped: block-scaled single-CTA tiles with one issuer");
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  if (base & 1023u) {  // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) record_status(a.status, FP8G_ERR_DEVICE_ASSERT);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // rank 0 of a pair issues the MMAs
  const uint32_t bar0 = base + C::kOffBar;
  auto full = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty = [&](uint32_t s) { return bar0 + 8u * (S + s); };
  constexpr uint32_t NB = C::kTmemBufs;
  // TMEM buffer b: partial written (tfull) / read (tempty)
  auto tfull = [&](uint32_t b) { return bar0 + 8u * (2 * S + b); };
  auto tempty = [&](uint32_t b) { return bar0 + 8u * (2 * S + NB + b); };
  const uint32_t xfull = bar0 + 8u * (2 * S + 2 * NB);  // K-split exchange written
  const uint32_t xempty = xfull + 8u;                             // K-split exchange read
  const uint32_t sk_written = xfull + 16u;  // stream-K: every epilogue warp has written its partial
  const uint32_t sk_ready = xfull + 24u;    // stream-K: the partials to add are complete
  // the scales of stage s have landed (K-grouped form)
  auto sfull = [&](uint32_t st) { return xfull + 32u + 8u * st; };
  // cluster K split: the partials of the other ranks are written (rank 0's barrier, ck - 1 arrivals)
  // (both recomputed from the kernel parameters where used, rather than kept in registers)
  auto ck_in = [&]() { return xfull + 32u + 8u * S; };
  auto ck_on = [&]() { return MODE == kDense && !PAIR && !EPI && a.ck > 1; };
  constexpr bool kStaged = MODE == kKGrouped;
  // Arrivals that free an operand stage: the MMA commit (lone issuers, CTA pairs and the
  // epilogue-scaled variant); else one lane of the promotion warps once the stage's MMAs have
  // completed (block forms), or every promotion warp once it has also read the stage's scales
  // (K-grouped).
  constexpr bool kCommitFrees = EPI || C::kMmaWarps > 1 || PAIR || C::kKPS > 1;
  constexpr uint32_t kEmptyArrivals = kCommitFrees ? 1u : (kStaged ? static_cast<uint32_t>(C::kEpiWarps) : 1u);
  // misc: [0] TMEM base, [1] abort flag, [2] group table out of contract
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  int32_t* table = reinterpret_cast<int32_t*>(smem + C::kOffTable);

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kEmptyArrivals);
      mbar_init(sfull(s), 1);  // the producer's expect-tx arrival
    }
    // each TMEM buffer is consumed by the warps of one K part (a stage-synchronised slot: by
    // every promotion warp)
    for (uint32_t b = 0; b < NB; ++b) {
      mbar_init(tfull(b), 1);
      // in a pair, the promotion warps of both CTAs release rank 0's buffer
      mbar_init(tempty(b), C::kStageSync ? C::kEpiWarps : (PAIR ? 2 * C::kStoreWarps : C::kStoreWarps));
    }
    mbar_init(xfull, C::kStoreWarps);
    mbar_init(xempty, C::kStoreWarps);
    mbar_init(sk_written, C::kEpiWarps);
    mbar_init(sk_ready, 1);
    mbar_init(ck_in(), ck_on() ? static_cast<uint32_t>(a.ck - 1) : 1u);
    misc[1] = 0;
    misc[2] = 0;  // set when the group table is out of contract
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmD);
    if (kStaged) {
      prefetch_tmap(&tmSA);
      prefetch_tmap(&tmSB);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // one warp of each CTA of the pair, collectively
      tmem_alloc_pair(base + C::kOffMisc, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(base + C::kOffMisc, C::kTmemCols);
      tmem_relinquish();
    }
  }
  // Everything above (barriers, TMEM, tensor-map prefetch) reads no input.  Launched as a
  // programmatic dependent of the kernel before it on the stream (a quantiser writing A), the
  // grid may have started early: wait for that kernel's results before the first input read.
  griddep_wait();
  // pair tiles per expert (prefix over experts), after the group table
  int32_t* ptab = table + (a.E + 1);
  // Group tables (grouped modes), built by the first epilogue warp.
  if ((MODE == kContiguous || MODE == kKGrouped) && warp == C::kEpiWarp0) {
    // offsets of rows (contiguous) or of tokens along K (K-grouped): multiples of 128, in range
    const int32_t limit = MODE == kKGrouped ? a.KB * BK : a.rows;
    bool bad = false;
    for (int i = lane; i <= a.E; i += 32) {
      const int32_t v = __ldg(a.groups + i);
      table[i] = v;
      if (v < 0 || (v & (BM - 1)) || v > limit) bad = true;
      if (i < a.E && __ldg(a.groups + i + 1) < v) bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) {
      misc[2] = 1;
      record_status(a.status, FP8G_ERR_DEVICE_ASSERT);
    }
    if constexpr (PAIR) {
      __syncwarp();
      int32_t running = 0;
      if (lane == 0) ptab[0] = 0;
      for (int e0 = 0; e0 < a.E; e0 += 32) {
        const int e = e0 + lane;
        int32_t prs = 0;
        if (e < a.E) prs = (max(table[e + 1] - table[e], 0) / BM + 1) >> 1;
        int32_t incl = prs;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        if (e < a.E) ptab[e + 1] = running + incl;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  if (MODE == kMasked && warp == C::kEpiWarp0) {
    int32_t running = 0;
    bool bad = false;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
      const int e = e0 + lane;
      int32_t mbs = 0;
      if (e < a.E) {
        const int32_t cnt = __ldg(a.groups + e);
        if (cnt < 0 || cnt > a.cap) bad = true;
        const int32_t c = min(max(cnt, 0), a.cap);
        mbs = (c + BM - 1) / BM;
        if (PAIR) mbs = (mbs + 1) >> 1;  // pair tiles
      }
      int32_t incl = mbs;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      if (e < a.E) (PAIR ? ptab : table)[e + 1] = running + incl;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) (PAIR ? ptab : table)[0] = 0;
    if (__any_sync(0xffffffffu, bad) && lane == 0) record_status(a.status, FP8G_ERR_DEVICE_ASSERT);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers and TMEM exist before any signalling
  if (ck_on()) cluster_sync();         // rank 0's barrier exists before the other ranks signal it
  tc_fence_after();
  const uint32_t tmem_base = misc[0];

  int32_t num_tiles = a.num_tiles;
  if (MODE == kMasked) num_tiles = (PAIR ? ptab : table)[a.E] * a.num_n;
  if (PAIR && MODE == kContiguous) num_tiles = ptab[a.E] * a.num_n;
  // a CTA pair walks the tiles of its cluster index; both CTAs see every pair tile
  const int32_t tile0 = PAIR ? static_cast<int32_t>(blockIdx.x >> 1) : static_cast<int32_t>(blockIdx.x);
  const int32_t tile_step = PAIR ? static_cast<int32_t>(gridDim.x >> 1) : static_cast<int32_t>(gridDim.x);
  // the tile of piece pc; K-grouped tiles cover their expert's K blocks (whole tiles only)
  auto fetch_tile = [&](Piece& pc, Tile& ti) -> bool {
    if constexpr (PAIR) {
      get_pair_tile<BN, MODE>(a, table, ptab, pc.t, rank, ti);
      return true;
    } else {
      const bool ok = get_tile<BN, MODE>(a, table, pc.t, ti);
      if (MODE == kKGrouped) pc.kb1 = ti.kb_count;
      return ok;
    }
  };
  if ((MODE == kContiguous || MODE == kKGrouped) && misc[2]) num_tiles = 0;
  // stream-K tail: single-CTA tiles with one K part and one issuer only
  const bool sk_on = !PAIR && C::kKSplit == 1 && C::kMmaWarps == 1 && a.sk != 0;
  if (warp < C::kEpiWarp0) {
    if constexpr (C::kRebalance) regs_release<C::kRegsLow>();
    const bool leader = lane == 0;
    constexpr int KPS = C::kKPS;
    constexpr int MW = C::kMmaWarps;
    // Lane 0 of the producer warp runs its loop alone.  One MMA issuer (wide tiles) runs its loop
    // with all 32 lanes (lane 0 issuing), each lane testing the barriers itself, without a warp
    // vote after each wait: measured per K block on 4096 x 8192 x 8192, ~850 cycles against ~900
    // with the vote and ~935 with lane 0 alone.  Two issuers (small-M tiles, 256 x 128 pair tiles)
    // run on lane 0 alone, test their next barriers ahead (wait_seen) and free stages by an MMA
    // commit; one issuer leaves the stage release to the promotion warps.
    constexpr bool kLone = MW > 1;
    static_assert(KPS == 1 || kCommitFrees, "multi-K-block stages are freed by the issuers' commits");
    // the tensor maps view A as [K/128][rows][128] and B as [E][K/128][N][128] (outer to
    // inner), so one box holds KPS K blocks of the tile's rows, K block by K block
    if (warp == 0 && leader) {
      // ---------------------------------------------------------- TMA producer
      uint32_t it = 0;  // stages filled
      bool ok = true;
      bool empty_seen = false;  // early test of the next stage's empty barrier (lone form)
      Work w = make_work(num_tiles, tile_step, tile0, a.KB, sk_on, a.sk_min_units, a.sk_min_gain, ck_on() ? a.ck : 0);
      Piece pc;
      while (ok && next_piece(w, pc)) {
        Tile ti;
        if (!fetch_tile(pc, ti)) continue;
        // the K blocks of a stage past the end of K are zero-filled and never read
        for (int32_t kb = pc.kb0; kb < pc.kb1; kb += KPS, ++it) {
          if (static_cast<int32_t>(it) == a.test_skip_stage) continue;  // test hook (see GemmArgs)
          const uint32_t s = it % S, ph = (it / S) & 1u;
          bool ready;
          if constexpr (kLone) {
            ready = wait_seen(empty_seen, empty(s), ph ^ 1u, a, abort_flag);
            empty_seen = mbar_test_wait(empty((it + 1) % S), (((it + 1) / S) & 1u) ^ 1u);
          } else {
            ready = wait_bounded(empty(s), ph ^ 1u, a, abort_flag);
          }
          if (!ready) { ok = false; break; }
          const uint32_t dA = base + C::kOffA + s * C::kStageABytes;
          const uint32_t dB = base + C::kOffB + s * C::kStageBBytes;
          if constexpr (PAIR) {
            // both CTAs' copies complete on rank 0's full barrier, which expects the pair's bytes
            const uint32_t fb = mapa_shared(full(s), 0);
            mbar_arrive_expect_tx(leader && rank == 0, full(s), 2 * (C::kStageABytes + C::kStageBBytes));
            tma_load_3d_pair(leader, dA, &tmA, fb, 0, ti.a_row, kb);
            tma_load_4d_pair(leader, dB, &tmB, fb, 0, ti.n0 + static_cast<int32_t>(rank) * C::kBRows, kb, ti.g);
          } else {
            mbar_arrive_expect_tx(leader, full(s), C::kStageABytes + C::kStageBBytes);
            tma_load_3d(leader, dA, &tmA, full(s), 0, ti.a_row, ti.kb_first + kb);
            tma_load_4d(leader, dB, &tmB, full(s), 0, ti.n0, ti.kb_first + kb, MODE == kKGrouped ? 0 : ti.g);
          }
          if constexpr (kStaged) {
            // the tile's A-row scales (rows past the matrix read as zero) and its per-column B scales
            const uint32_t dS = base + C::kOffScale + s * C::kScaleStage;
            mbar_arrive_expect_tx(leader, sfull(s), C::kSAKB + C::kSBKB);
            tma_load_2d(leader, dS, &tmSA, sfull(s), ti.a_row, ti.kb_first + kb);
            tma_load_2d(leader, dS + C::kSAKB, &tmSB, sfull(s), ti.n0, ti.kb_first + kb);
          }
        }
      }
      if (!ok && leader && rank == 0) {  // let the loads already issued land before the CTA exits
        const uint32_t n = it < S ? it : S;
        for (uint32_t i = it - n; i < it; ++i) {
          const long long t0 = clock64();
          while (!mbar_try_wait(full(i % S), (i / S) & 1u) && clock64() - t0 < a.budget) {
          }
        }
      }
    } else if (warp >= 1 && warp <= MW && rank == 0 && (!kLone || leader)) {
      // ---------------------------------------------------------- MMA issuer(s) (rank 0 of a pair)
      const uint32_t idesc = idesc_e4m3_f32(PAIR ? 2 * BM : BM, BN) | a.idesc_fmt;
      // descriptors of stage 0; stage s and K step k add (offset in bytes) / 16 to the
      // 14-bit start-address field (shared addresses stay below 2^18, so it cannot carry)
      const uint64_t adesc0 = smem_desc_k_sw128(base + C::kOffA);
      const uint64_t bdesc0 = smem_desc_k_sw128(base + C::kOffB);
      if constexpr (EPI) {
        // one TMEM accumulator per piece, all its K blocks accumulated in place; the commit after
        // a K block's MMAs frees its stage, the commit after the last one hands the buffer over
        uint32_t it = 0, np = 0;
        bool ok = true;
        Work w = make_work(num_tiles, tile_step, tile0, a.KB, sk_on, a.sk_min_units, a.sk_min_gain, ck_on() ? a.ck : 0);
        Piece pc;
        while (ok && next_piece(w, pc)) {
          Tile ti;
          if (!fetch_tile(pc, ti)) continue;
          const uint32_t b = np % NB, tph = (np / NB) & 1u;
          ++np;
          if (!(wait_bounded(tempty(b), tph ^ 1u, a, abort_flag))) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * C::kTmemStride;
          for (int32_t kb = pc.kb0; kb < pc.kb1; ++kb, ++it) {
            const uint32_t s = it % S, ph = (it / S) & 1u;
            if (!(wait_bounded(full(s), ph, a, abort_flag))) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = adesc0 + ((s * C::kStageABytes) >> 4);
            const uint64_t bd = bdesc0 + ((s * C::kStageBBytes) >> 4);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              mma_f8f6f4(leader, d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb > pc.kb0 || k > 0) ? 1u : 0u);
            mma_commit(leader, empty(s));
          }
          if (!ok) break;
          mma_commit(leader, tfull(b));
        }
        if (!ok && it > 0 && leader) {  // the last stage commit completes after every issued MMA
          const uint32_t last = it - 1;
          const long long t0 = clock64();
          while (!mbar_try_wait(empty(last % S), (last / S) & 1u) && clock64() - t0 < a.budget) {
          }
        }
      } else if constexpr (!kLone) {
        // stage `it` holds the K blocks kb .. kb + nk - 1 of the piece (nk = min(KPS, K blocks
        // left in it)); `kit` counts K blocks, the TMEM buffer sequence as the epilogue counts it
        uint32_t it = 0, kit = 0;
        bool ok = true;
        Work w = make_work(num_tiles, tile_step, tile0, a.KB, sk_on, a.sk_min_units, a.sk_min_gain, ck_on() ? a.ck : 0);
        Piece pc;
        while (ok && next_piece(w, pc)) {
          Tile ti;
          if (!fetch_tile(pc, ti)) continue;
          for (int32_t kb = pc.kb0; kb < pc.kb1; kb += KPS, ++it) {
            const uint32_t s = it % S, ph = (it / S) & 1u;
            // the operand stage first: it is nearly always complete, and testing it costs a round
            // trip that would otherwise sit between the buffer's release and the MMAs
            if (!(wait_bounded(full(s), ph, a, abort_flag))) { ok = false; break; }
            const int32_t nk = min(KPS, pc.kb1 - kb);
            for (int32_t j = 0; j < nk; ++j, ++kit) {
              const uint32_t b = kit % NB, tph = (kit / NB) & 1u;
              if (!(wait_bounded(tempty(b), tph ^ 1u, a, abort_flag))) { ok = false; break; }
              tc_fence_after();
              const uint64_t ad = adesc0 + ((s * C::kStageABytes + j * C::kABytes) >> 4);
              const uint64_t bd = bdesc0 + ((s * C::kStageBBytes + j * C::kBBytes) >> 4);
              const uint32_t d_tmem = tmem_base + b * C::kTmemStride;
              if constexpr (PAIR) {
#pragma unroll
                for (int k = 0; k < BK / 32; ++k)
                  mma_f8f6f4_pair(leader, d_tmem, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                mma_commit_pair(leader, empty(s), 0x3);  // both CTAs' stage s is free
                mma_commit_pair(leader, tfull(b), 0x3);  // both CTAs' partial is ready
              } else {
#pragma unroll
                for (int k = 0; k < BK / 32; ++k)
                  mma_f8f6f4(leader, d_tmem, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                // one commit per K block; with one K block per stage the promotion warps free the
                // stage once it has completed
                mma_commit(leader, tfull(b));
              }
            }
            if (!ok) break;
            if constexpr (KPS > 1) mma_commit(leader, empty(s));  // the stage's MMAs have read it
          }
        }
        if (!ok && kit > 0 && leader) {  // wait for the MMAs already issued before TMEM is released
          const uint32_t last = kit - 1;
          const long long t0 = clock64();
          while (!mbar_try_wait(tfull(last % NB), (last / NB) & 1u) && clock64() - t0 < a.budget) {
          }
        }
      } else {
        // Lone issuers: issuer mi takes the stages it % MW == mi.  Stage `it` (counted over this
        // CTA's tiles) holds the K blocks kb0 .. kb0 + nk - 1 of its tile, nk = min(KPS, K blocks
        // left); `kit` counts the K blocks of all earlier stages (the TMEM buffer sequence, as
        // the epilogue counts them).
        static_assert(MW == 2 || C::kStageSync, "two lone issuers (stage-synchronised tiles: any number)");
        const uint32_t mi = static_cast<uint32_t>(warp - 1);
        uint32_t it = 0, kit = 0;
        bool ok = true, issued = false;
        uint32_t last_bar = 0, last_ph = 0;  // latest commit to a TMEM-full barrier
        bool full_seen = false, tmem_seen = false;  // early tests for the next own K block
        Work w = make_work(num_tiles, tile_step, tile0, a.KB, false, 0, 0);  // whole tiles
        Piece pc;
        if constexpr (C::kStageSync) {
          // stage `it` fills TMEM slot it % NSL (its K block j in buffer j of the slot): one wait
          // for the slot, one commit for its partials, one for the operand stage
          constexpr uint32_t NSL = C::kTmemSlots;
          while (ok && next_piece(w, pc)) {
            Tile ti;
            if (!fetch_tile(pc, ti)) continue;
            for (int32_t kb0 = 0; kb0 < a.KB; kb0 += KPS, ++it) {
              if (it % MW != mi) continue;
              const int32_t left = a.KB - kb0;
              const uint32_t nk = static_cast<uint32_t>(left < KPS ? left : KPS);
              const uint32_t s = it % S, ph = (it / S) & 1u;
              const uint32_t sl = it % NSL, tph = (it / NSL) & 1u;
              if (!wait_seen(full_seen, full(s), ph, a, abort_flag)) { ok = false; break; }
              if (!wait_seen(tmem_seen, tempty(sl), tph ^ 1u, a, abort_flag)) { ok = false; break; }
              tc_fence_after();
              // test the next own stage's barriers now; the MMAs below hide the round trips.  Neither
              // test can take an older phase for this one: stage nx - S is this issuer's own (S is a
              // multiple of MW) and already consumed, so its fill has landed; and every warp releases
              // stages in order, so the release of stage nx - 2 NSL came before that of stage
              // it - NSL, awaited above.
              const uint32_t nx = it + MW;
              full_seen = mbar_test_wait(full(nx % S), (nx / S) & 1u);
              tmem_seen = mbar_test_wait(tempty(nx % NSL), ((nx / NSL) & 1u) ^ 1u);
              for (uint32_t j = 0; j < nk; ++j) {
                const uint64_t ad = adesc0 + ((s * C::kStageABytes + j * C::kABytes) >> 4);
                const uint64_t bd = bdesc0 + ((s * C::kStageBBytes + j * C::kBBytes) >> 4);
                const uint32_t d_tmem = tmem_base + sl * C::kSlotCols + j * C::kTmemStride;
#pragma unroll
                for (int k = 0; k < BK / 32; ++k)
                  mma_f8f6f4(true, d_tmem, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
              }
              mma_commit(true, tfull(sl));
              mma_commit(true, empty(s));  // the stage is free once these MMAs have read it
              issued = true;
              last_bar = tfull(sl);
              last_ph = tph;
            }
          }
        }
        while (!C::kStageSync && ok && next_piece(w, pc)) {
          Tile ti;
          if (!fetch_tile(pc, ti)) continue;
          for (int32_t kb0 = 0; kb0 < a.KB && ok; kb0 += KPS, ++it) {
            const int32_t left = a.KB - kb0;
            const uint32_t nk = static_cast<uint32_t>(left < KPS ? left : KPS);
            if (it % MW == mi) {
              const uint32_t s = it % S, ph = (it / S) & 1u;
              if (!wait_seen(full_seen, full(s), ph, a, abort_flag)) { ok = false; break; }
              full_seen = false;
              for (uint32_t j = 0; j < nk; ++j) {
                const uint32_t kj = kit + j;
                const uint32_t b = kj % NB, tph = (kj / NB) & 1u;
                if (!wait_seen(tmem_seen, tempty(b), tph ^ 1u, a, abort_flag)) { ok = false; break; }
                tc_fence_after();
                // test the next own K block's barriers now; the MMAs below hide the round trip
                uint32_t kn = kj + 1;
                if (j + 1 == nk) {  // the next own K block opens stage it + MW, past the other
                                    // issuer's stage (which may start the next tile)
                  const int32_t p = kb0 + KPS < a.KB ? kb0 + KPS : 0;
                  kn += static_cast<uint32_t>(a.KB - p < KPS ? a.KB - p : KPS);
                  full_seen = mbar_test_wait(full((it + MW) % S), ((it + MW) / S) & 1u);
                }
                tmem_seen = mbar_test_wait(tempty(kn % NB), ((kn / NB) & 1u) ^ 1u);
                const uint64_t ad = adesc0 + ((s * C::kStageABytes + j * C::kABytes) >> 4);
                const uint64_t bd = bdesc0 + ((s * C::kStageBBytes + j * C::kBBytes) >> 4);
                const uint32_t d_tmem = tmem_base + b * C::kTmemStride;
                if constexpr (PAIR) {  // rank 0 issues for the pair; both CTAs' partials are ready
#pragma unroll
                  for (int k = 0; k < BK / 32; ++k)
                    mma_f8f6f4_pair(true, d_tmem, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                  mma_commit_pair(true, tfull(b), 0x3);
                } else {
#pragma unroll
                  for (int k = 0; k < BK / 32; ++k)
                    mma_f8f6f4(true, d_tmem, ad + 2 * k, bd + 2 * k, idesc, k > 0 ? 1u : 0u);
                  mma_commit(true, tfull(b));
                }
                issued = true;
                last_bar = tfull(b);
                last_ph = tph;
              }
              if (!ok) break;
              // the stage is free once these MMAs have read it (in a pair: both CTAs' stages)
              if constexpr (PAIR) mma_commit_pair(true, empty(s), 0x3);
              else mma_commit(true, empty(s));
            }
            kit += nk;
          }
        }
        if (!ok && issued) {  // wait for the MMAs already issued before TMEM is released
          const long long t0 = clock64();
          while (!mbar_try_wait(last_bar, last_ph) && clock64() - t0 < a.budget) {
          }
        }
      }
    }
    __syncwarp();  // the other lanes of the producer and MMA warps wait for lane 0 here
  } else {
    if constexpr (C::kRebalance) regs_acquire<C::kRegsHigh>();
    // ------------------------------------------------------------ promotion + epilogue
    const int ew = warp - C::kEpiWarp0;  // epilogue warp index
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int grp = ew >> 2;             // epilogue warpgroup
    const int kpart = grp / C::kColGroups;                 // promotes K blocks kb % kKSplit == kpart
    const int col0 = (grp % C::kColGroups) * C::kEpiCols;  // column offset inside the tile
    const int row = q * 32 + lane;       // tile row owned by this thread
    // this warp's TMEM buffers are released on rank 0's barrier (its own CTA unless paired)
    auto release_tmem = [&](uint32_t b) {
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_remote(mapa_shared(tempty(b), 0));
        else mbar_arrive(tempty(b));
      }
    };
    const uint32_t out_addr = base + C::kOffOut + (ew % C::kStoreWarps) * C::kOutWarpBytes;
    const uint32_t sbv_addr = base + C::kOffSbv + ew * 512u;  // K-grouped: this warp's B scales
    float2* xbuf = reinterpret_cast<float2*>(smem + C::kOffX);
    uint32_t it_base = 0, tiles_done = 0;
    uint32_t st_base = 0;  // stages of earlier pieces (stage-synchronised TMEM slots)
    uint32_t np = 0;  // pieces taken (EPI: the TMEM buffer sequence, as the MMA warp counts it)
    bool ok = true;
    // stream-K workspace slot of this thread: float4 j of thread e sits at slot[j * kEpiThreads + e]
    constexpr int kEpiThreads = C::kEpiWarps * 32;
    constexpr int64_t kSlotF4 = static_cast<int64_t>(kEpiThreads) * (C::kEpiCols / 4);
    const int e_thr = ew * 32 + lane;
    Work w = make_work(num_tiles, tile_step, tile0, a.KB, sk_on, a.sk_min_units, a.sk_min_gain, ck_on() ? a.ck : 0);
    Piece pc;
    while (ok && next_piece(w, pc)) {
      Tile ti;
      if (!fetch_tile(pc, ti)) continue;
      const int32_t ncol0 = ti.n0 + col0;
      const bool has_cols = ncol0 < a.N;
      // small-M tiles: warps whose rows are all past M skip the promotion (nothing to store)
      const bool live = (MODE != kDenseSmallM && !PAIR) || q * 32 < ti.rows;
      const int32_t grow = ti.a_row + row;
      const bool row_ok = grow < a.rows;
      float2 acc[C::kEpiCols / 2];
      if constexpr (EPI) {
        // the tile's accumulator, read once
        const uint32_t b = np % NB, tph = (np / NB) & 1u;
        ++np;
        if (!__all_sync(0xffffffffu, wait_bounded(tfull(b), tph, a, abort_flag))) { ok = false; break; }
        tc_fence_after();
        if (live) {
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * C::kTmemStride + col0;
#pragma unroll
          for (int c = 0; c < C::kEpiCols / 64; ++c) {
            float v[64];
            tmem_ld64_sync(taddr + c * 64, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[c * 32 + i] = make_float2(v[2 * i], v[2 * i + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        release_tmem(b);
      } else if constexpr (MODE == kSwapAB) {
        // D^T tile: this thread's row is weight row `grow`, its columns the tokens ncol0 .. +31.
        // Per K block acc += P * (sw * sa[m]): sw the scale of the tile's 128 x 128 weight block (one
        // per tile), sa[m] the tokens' scales (one per column, the same for every thread: broadcast
        // loads).  Both come from global memory two K-block steps ahead, in two register sets used
        // alternately (the loop below is unrolled by two, as in the block forms).
        constexpr int NC = C::kEpiCols;
        static_assert(NC == 32 && C::kKSplit == 1, "swapped tiles: 32 columns a warp");
#pragma unroll
        for (int j = 0; j < NC / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
        const float* swp = a.sB + static_cast<int64_t>(ti.a_row / BM) * a.KB;
        const float* scp = a.sA + ncol0;
        const int32_t ncv = a.N - ncol0;  // token columns of this warp that exist
        auto load_sc = [&](int32_t kbi, float (&c)[NC], float& w) {
          const bool in = kbi < pc.kb1;
          w = ld_nc_f32_or0(swp + kbi, in);
          const float* p = scp + static_cast<int64_t>(kbi) * a.ld_sa;
          if (in && ncv >= NC) {  // (16-byte aligned: ld_sa and ncol0 are multiples of 4)
#pragma unroll
            for (int j = 0; j < NC / 4; ++j) {
              const float4 t = __ldg(reinterpret_cast<const float4*>(p) + j);
              c[4 * j] = t.x;
              c[4 * j + 1] = t.y;
              c[4 * j + 2] = t.z;
              c[4 * j + 3] = t.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < NC; ++j) c[j] = ld_nc_f32_or0(p + j, in && j < ncv);
          }
        };
        float c0[NC], c1[NC], w0, w1;
        load_sc(pc.kb0, c0, w0);
        load_sc(pc.kb0 + 1, c1, w1);
        auto step = [&](int32_t kb, float (&c)[NC], float& w) -> bool {
          const uint32_t it = it_base + static_cast<uint32_t>(kb - pc.kb0);
          const uint32_t b = it % NB, tph = (it / NB) & 1u;
          if (!__all_sync(0xffffffffu, wait_bounded(tfull(b), tph, a, abort_flag))) return false;
          tc_fence_after();
          float v[NC];
          tmem_ld32_sync(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * C::kTmemStride + col0, v);
          tc_fence_before();
          __syncwarp();
          release_tmem(b);
          const float2 w2 = make_float2(w, w);
#pragma unroll
          for (int j = 0; j < NC / 2; ++j)
            acc[j] = __ffma2_rn(make_float2(v[2 * j], v[2 * j + 1]),
                                __fmul2_rn(make_float2(c[2 * j], c[2 * j + 1]), w2), acc[j]);
          load_sc(kb + 2, c, w);  // these registers' next use is two steps on
          return true;
        };
        for (int32_t kb = pc.kb0; kb < pc.kb1; kb += 2) {
          if (!step(kb, c0, w0)) { ok = false; break; }
          if (kb + 1 >= pc.kb1) break;
          if (!step(kb + 1, c1, w1)) { ok = false; break; }
        }
      } else {
        // Per K block: acc += P * (sa * sb), with the partial P from TMEM.
        //   Block forms: sa (this thread's row) and sb (this warp's 128-column block) come from
        //   global memory two K-block steps ahead of use, in two register pairs used alternately:
        //   the loop below is unrolled by two, so a pair is touched only by its load and, two
        //   steps later, its use (no wait on a load in between, and no barrier or shared-memory
        //   round trip per K block).
        //   K-grouped: sa and the per-column B scales from the stage's scales in shared memory.
#pragma unroll
        for (int j = 0; j < C::kEpiCols / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
        constexpr int KS = C::kKSplit;
        const float* sap = a.sA + static_cast<int64_t>(ti.kb_first) * a.ld_sa + grow;
        const float* sbp = a.sB + (static_cast<int64_t>(ti.g) * a.NBs + ncol0 / 128) * a.KB;
        const bool blk_sb = MODE != kKGrouped && has_cols;
        // 48-wide tiles may straddle a 128-column weight block: its columns from `cut` on take the
        // next block's scale (cut is a multiple of 16, so a column pair never straddles it)
        constexpr bool kTwoSb = C::kEpiCols == 48;
        const int32_t cut = kTwoSb ? 128 - ncol0 % 128 : C::kEpiCols;
        const bool has_hi = kTwoSb && cut < C::kEpiCols && ncol0 / 128 + 1 < a.NBs;
        auto load_scales = [&](int32_t kbi, float& sa_o, float& sb_o, float& sbh_o) {
          sa_o = ld_nc_f32_or0(sap + static_cast<int64_t>(kbi) * a.ld_sa, MODE != kKGrouped && row_ok && kbi < pc.kb1);
          sb_o = ld_nc_f32_or0(sbp + kbi, blk_sb && kbi < pc.kb1);
          sbh_o = kTwoSb ? ld_nc_f32_or0(sbp + a.KB + kbi, blk_sb && has_hi && kbi < pc.kb1) : 0.0f;
        };
        float sa0, sb0, sbh0, sa1, sb1, sbh1;
        load_scales(pc.kb0 + kpart, sa0, sb0, sbh0);
        load_scales(pc.kb0 + kpart + KS, sa1, sb1, sbh1);
        // What sets the pace of the wide tiles: a TMEM buffer is written again (K block kb + NB)
        // only after all of its warps have loaded it, so each K block's MMA, its completion, these
        // loads and the release form a chain that NB = 2 buffers must cover.
        auto step = [&](int32_t kb, float& sa_r, float& sb_r, float& sbh_r) -> bool {
          const uint32_t it = it_base + static_cast<uint32_t>(kb - pc.kb0);
          // the barrier pair, its phase and the TMEM columns of this K block's partial
          uint32_t b = it % NB, tph = (it / NB) & 1u, tcol = b * C::kTmemStride;
          if constexpr (C::kStageSync) {
            const uint32_t r = static_cast<uint32_t>(kb - pc.kb0);
            const uint32_t st = st_base + r / C::kKPS;
            b = st % C::kTmemSlots;
            tph = (st / C::kTmemSlots) & 1u;
            tcol = b * C::kSlotCols + (r % C::kKPS) * C::kTmemStride;
          }
          const uint32_t s = it % S, sph = (it / S) & 1u;  // (one K block per stage)
          float sa_kb = sa_r, sb_kb = sb_r;
          const float sbh_kb = sbh_r;
          load_scales(kb + 2 * KS, sa_r, sb_r, sbh_r);
          if constexpr (MODE == kKGrouped) {
            // the stage's scales land long before its partial: take them first
            if (!__all_sync(0xffffffffu, wait_bounded(sfull(s), sph, a, abort_flag))) return false;
            const uint32_t sc = base + C::kOffScale + s * C::kScaleStage;
            sa_kb = ld_shared_f32(sc + 4u * static_cast<uint32_t>(row));
            // lane l: the B scales of columns col0 + 4l .. 4l+3, copied into this warp's own area
            const float4 v = ld_shared_v4f(sc + C::kSAKB + 4u * static_cast<uint32_t>(col0) + 16u * lane);
            __syncwarp();  // every lane has read the previous K block's copy
            st_shared_v4(sbv_addr + 16 * lane, __float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                         __float_as_uint(v.w));
            __syncwarp();
          }
          const float scale = sa_kb * sb_kb;
          const float2 scale2 = make_float2(scale, scale);
          const float scale_hi = sa_kb * sbh_kb;
          const float2 scale2_hi = make_float2(scale_hi, scale_hi);
          if (!__all_sync(0xffffffffu, wait_bounded(tfull(b), tph, a, abort_flag))) return false;
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + tcol + col0;
          if (live) {
            // this warp's columns in loads of kLd (one load and its wait each)
            constexpr int kLd = C::kEpiCols >= 64 ? 64 : C::kEpiCols;
#pragma unroll
            for (int c = 0; c < C::kEpiCols / kLd; ++c) {
              float v[kLd];
              tmem_ld_sync(taddr + c * kLd, v);
              if (c == C::kEpiCols / kLd - 1) {  // all of this warp's columns are in registers:
                tc_fence_before();                // release the TMEM buffer before the last FMAs
                __syncwarp();
                release_tmem(b);
              }
              if constexpr (MODE == kKGrouped) {
                static_assert(MODE != kKGrouped || kLd == 64, "K-grouped tiles load 64 columns at a time");
                // one B scale per column: s[n] = sa * sB[kb][n]
                const float2 sa2 = make_float2(sa_kb, sa_kb);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float4 s4 = ld_shared_v4f(sbv_addr + 16 * (c * 16 + i));
                  const float2 s01 = __fmul2_rn(sa2, make_float2(s4.x, s4.y));
                  const float2 s23 = __fmul2_rn(sa2, make_float2(s4.z, s4.w));
                  acc[c * 32 + 2 * i] = __ffma2_rn(make_float2(v[4 * i], v[4 * i + 1]), s01, acc[c * 32 + 2 * i]);
                  acc[c * 32 + 2 * i + 1] =
                      __ffma2_rn(make_float2(v[4 * i + 2], v[4 * i + 3]), s23, acc[c * 32 + 2 * i + 1]);
                }
              } else if constexpr (kTwoSb) {
#pragma unroll
                for (int i = 0; i < kLd / 2; ++i)
                  acc[i] = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), 2 * i < cut ? scale2 : scale2_hi, acc[i]);
              } else {
#pragma unroll
                for (int i = 0; i < kLd / 2; ++i)
                  acc[c * (kLd / 2) + i] =
                      __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), scale2, acc[c * (kLd / 2) + i]);
              }
            }
          } else {
            tc_fence_before();
            __syncwarp();
            release_tmem(b);
          }
          // Free the operand stage (one K block per stage in these forms) once its MMAs are known
          // complete -- here, after the TMEM release, off the path from the partial to the next
          // MMAs.  K-grouped: every warp, having read the stage's scales; else the first warp of
          // each K part (lone issuers, pairs and the epilogue-scaled variant free stages by commit).
          if constexpr (!kCommitFrees) {
            if (lane == 0 && (kStaged || ew == kpart * 4 * C::kColGroups)) mbar_arrive(empty(s));
          }
          return true;
        };
        for (int32_t kb = pc.kb0 + kpart; kb < pc.kb1; kb += 2 * KS) {
          if (!step(kb, sa0, sb0, sbh0)) { ok = false; break; }
          if (kb + KS >= pc.kb1) break;
          if (!step(kb + KS, sa1, sb1, sbh1)) { ok = false; break; }
        }
        if constexpr (C::kStageSync) {
          // a last stage holding fewer K blocks than K parts: the warps of the K parts without
          // one release its slot too, once its partials have been written (so that the release
          // is counted in that phase, not an earlier one)
          const int32_t n = pc.kb1 - pc.kb0;
          if (ok && n % C::kKPS != 0 && kpart >= n % C::kKPS) {
            const uint32_t st = st_base + static_cast<uint32_t>(n - 1) / C::kKPS;
            const uint32_t b = st % C::kTmemSlots;
            if (!__all_sync(0xffffffffu, wait_bounded(tfull(b), (st / C::kTmemSlots) & 1u, a, abort_flag))) {
              ok = false;
            } else {
              __syncwarp();
              release_tmem(b);
            }
          }
        }
      }
      it_base += static_cast<uint32_t>(pc.kb1 - pc.kb0);
      st_base += static_cast<uint32_t>(pc.kb1 - pc.kb0 + C::kKPS - 1) / C::kKPS;
      if (!ok) break;
      if constexpr (C::kKSplit > 1) {
        // add the odd-K-block partial sums (second warpgroup) into the first warpgroup's
        const uint32_t xph = tiles_done & 1u;
        ++tiles_done;
        if (kpart == 1) {
          if (!__all_sync(0xffffffffu, wait_bounded(xempty, xph ^ 1u, a, abort_flag))) { ok = false; break; }
          if (live) {
#pragma unroll
            for (int i = 0; i < C::kEpiCols / 2; ++i) xbuf[i * C::kXRows + row] = acc[i];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(xfull);
          continue;
        }
        if (!__all_sync(0xffffffffu, wait_bounded(xfull, xph, a, abort_flag))) { ok = false; break; }
        if (live) {
#pragma unroll
          for (int i = 0; i < C::kEpiCols / 2; ++i) {
            const float2 o = xbuf[i * C::kXRows + row];
            acc[i].x += o.x;
            acc[i].y += o.y;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(xempty);
      }
      if (pc.kind == kContrib) {
        // part of a split tile: the FP32 partial goes to this CTA's workspace slot (L2), then
        // the flag is raised once every epilogue warp has written its share (cluster K split:
        // rank 0's barrier is signalled instead)
        // (warps whose rows are all past the matrix skip it, and the finishing CTA skips them too)
        float4* slot = a.ws_part + static_cast<int64_t>(blockIdx.x) * kSlotF4;
        if (ti.a_row + q * 32 < a.rows) {
#pragma unroll
          for (int j = 0; j < C::kEpiCols / 4; ++j)
            __stcg(slot + static_cast<int64_t>(j) * kEpiThreads + e_thr,
                   make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x, acc[2 * j + 1].y));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(sk_written);
        if (ew == 0 && lane == 0 && wait_bounded(sk_written, 0u, a, abort_flag)) {
          if (ck_on()) {  // signal rank 0 of the cluster (release at cluster scope)
            fence_acq_rel_cluster();
            mbar_arrive_remote(mapa_shared(ck_in(), 0));
          } else {
            st_release_gpu(a.ws_flag + blockIdx.x, 1u);
          }
        }
        continue;
      }
      if (pc.kind == kFinish) {
        // first K blocks of a split tile: add the partials of CTAs c_lo .. c_hi once their
        // flags are up, or (cluster K split) once they have signalled this CTA's barrier (one
        // thread waits; it releases the others even on a timeout)
        if (ew == 0 && lane == 0) {
          if (ck_on()) {
            if (wait_bounded(ck_in(), 0u, a, abort_flag)) fence_acq_rel_cluster();
          } else {
            bool got = true;
            for (int32_t c2 = pc.c_lo; c2 <= pc.c_hi && got; ++c2) got = wait_flag(a.ws_flag + c2, a, abort_flag);
          }
          mbar_arrive(sk_ready);
        }
        if (!__all_sync(0xffffffffu, wait_bounded(sk_ready, 0u, a, abort_flag))) { ok = false; break; }
        for (int32_t c2 = pc.c_lo; c2 <= pc.c_hi && ti.a_row + q * 32 < a.rows; ++c2) {
          const float4* slot = a.ws_part + static_cast<int64_t>(c2) * kSlotF4;
#pragma unroll
          for (int j = 0; j < C::kEpiCols / 4; ++j) {
            const float4 v = __ldcg(slot + static_cast<int64_t>(j) * kEpiThreads + e_thr);
            acc[2 * j].x += v.x;
            acc[2 * j].y += v.y;
            acc[2 * j + 1].x += v.z;
            acc[2 * j + 1].y += v.w;
          }
        }
      }
      // ---- epilogue: this warp holds rows q*32 .. q*32+31, columns ncol0 .. ncol0+kEpiCols-1
      const int nvalid = min(32, ti.rows - q * 32);
      if (nvalid <= 0 || !has_cols) continue;
      if constexpr (MODE == kSwapAB) {
        // transposed: D[m][n] for this thread's weight row n and the warp's tokens m; for a fixed
        // token the 32 lanes write 32 consecutive bf16 of that row of D (64 bytes)
        if (row_ok) {
          __nv_bfloat16* dcol = a.D + grow;
          const int32_t nv = min(C::kEpiCols, a.N - ncol0);
#pragma unroll
          for (int j = 0; j < C::kEpiCols; ++j) {
            if (j < nv)
              dcol[static_cast<int64_t>(ncol0 + j) * a.ldd] =
                  __float2bfloat16_rn((j & 1) ? acc[j >> 1].y : acc[j >> 1].x);
          }
        }
        continue;
      }
      if constexpr (EPI) {
        // D = bf16(acc * fp32(sa[m] * sb[n])); sb is read with warp-uniform addresses (broadcast)
        const float sa_r = row_ok ? ld_nc_f32(a.sA + (a.sa_step ? grow : 0)) : 0.0f;
        if (a.sb_step) {
          const float* sbp = a.sB + static_cast<int64_t>(ti.g) * a.N + ncol0;
#pragma unroll
          for (int j = 0; j < C::kEpiCols / 4; ++j) {
            if (ncol0 + 4 * j < a.N) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(sbp) + j);
              acc[2 * j] = __fmul2_rn(acc[2 * j], make_float2(__fmul_rn(sa_r, v.x), __fmul_rn(sa_r, v.y)));
              acc[2 * j + 1] = __fmul2_rn(acc[2 * j + 1], make_float2(__fmul_rn(sa_r, v.z), __fmul_rn(sa_r, v.w)));
            }
          }
        } else {
          const float sc = __fmul_rn(sa_r, ld_nc_f32(a.sB + ti.g));
#pragma unroll
          for (int j = 0; j < C::kEpiCols / 2; ++j) acc[j] = __fmul2_rn(acc[j], make_float2(sc, sc));
        }
      }
      // (48-wide tiles take the plain stores: a 32-column box would spill into the next tile)
      if (C::kEpiCols % 32 == 0 && ((MODE != kMasked && MODE != kKGrouped) || nvalid == 32)) {
#pragma unroll
        for (int j = 0; j < C::kEpiCols / 32; ++j) {
          if (ncol0 + 32 * j >= a.N) break;
          // the staging box has left for global memory: with one box per warp, the previous box;
          // with a box per 32 columns (K-grouped), the previous tile's boxes
          const uint32_t box = out_addr + (C::kOutBoxes > 1 ? j * C::kOutBytes : 0u);
          if (C::kOutBoxes == 1 || j == 0) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(acc[16 * j + i].x, acc[16 * j + i].y);
          const uint32_t rowaddr = box + lane * 64;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            // 64-byte swizzle: 16-byte chunk index XOR address bits 7-8 (= row / 2 mod 4)
            st_shared_v4(rowaddr + ((ch ^ ((lane >> 1) & 3)) << 4), p[4 * ch], p[4 * ch + 1],
                         p[4 * ch + 2], p[4 * ch + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmD, box, ncol0 + 32 * j, ti.d_row + q * 32);
            bulk_commit();
          }
        }
      } else if (lane < nvalid) {
        // partial rows (a masked expert's count, the last rows of a K-grouped expert's matrix, the
        // small-M tiles' rows up to M) and 48-wide tiles: plain stores, row by row
        __nv_bfloat16* drow = a.D + static_cast<int64_t>(ti.d_row + q * 32 + lane) * a.ldd + ncol0;
#pragma unroll
        for (int j = 0; j < C::kEpiCols / 8; ++j) {
          if (ncol0 + 8 * j < a.N) {
            uint4 v;
            v.x = pack_bf16x2(acc[4 * j + 0].x, acc[4 * j + 0].y);
            v.y = pack_bf16x2(acc[4 * j + 1].x, acc[4 * j + 1].y);
            v.z = pack_bf16x2(acc[4 * j + 2].x, acc[4 * j + 2].y);
            v.w = pack_bf16x2(acc[4 * j + 3].x, acc[4 * j + 3].y);
            *reinterpret_cast<uint4*>(drow + 8 * j) = v;
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
  if (ck_on()) cluster_sync();         // rank 0 leaves after every rank has signalled it
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Self-test of the bounded waits the GEMM's roles use: one thread waits on an mbarrier phase that
// nothing completes, then on a global flag that nothing raises.  Nothing is in flight, so each wait
// can only run out of its budget; each must then record FP8G_ERR_TIMEOUT and return false.
// out[0] / out[1]: 1 when the mbarrier / flag wait returned false, out[2]: the abort flag.
__device__ uint32_t g_never_raised = 0u;

__global__ void bounded_wait_selftest_kernel(const GemmArgs a, uint32_t* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  volatile int* abort_flag = &abort_word;
  *abort_flag = 0;
  const bool bar_ok = wait_bounded(smem_u32(&bar), 0u, a, abort_flag);  // phase 0: no arrival
  const int abort_after_bar = *abort_flag;
  *abort_flag = 0;
  const bool flag_ok = wait_flag(&g_never_raised, a, abort_flag);
  out[0] = bar_ok ? 0u : 1u;
  out[1] = flag_ok ? 0u : 1u;
  out[2] = static_cast<uint32_t>(abort_after_bar && *abort_flag);
}

// ---------------------------------------------------------------- host side

template <int BN, bool SMALL = false, bool PAIR = false, bool KG = false, bool SWAP = false>
constexpr uint32_t smem_bytes(int table_entries) {
  return Cfg<BN, SMALL, PAIR, KG, SWAP>::kOffTable + ((table_entries * 4 + 15) / 16) * 16;
}

constexpr int kMaxExperts = 2048;
constexpr uint32_t kSmemLimit = 232448;  // 227 KB: the per-block dynamic shared memory limit
static_assert(Cfg<256>::kOffTable + 4 * (kMaxExperts + 1) <= kSmemLimit, "smem");
static_assert(Cfg<128>::kOffTable + 4 * (kMaxExperts + 1) <= kSmemLimit, "smem");
static_assert(Cfg<192>::kOffTable + 4 * (kMaxExperts + 1) <= kSmemLimit, "smem");
// 160-wide tiles (four 36 KB stages and twenty 2 KB staging boxes) leave room for the group tables
// of up to 512 experts; grouped calls with more experts take 256-wide tiles.
constexpr int kMaxExperts160 = 512;
static_assert(Cfg<160>::kOffTable + 4 * (kMaxExperts160 + 1) <= kSmemLimit, "smem");
static_assert(Cfg<64>::kOffTable + 4 * (kMaxExperts + 1) <= kSmemLimit, "smem");
static_assert(Cfg<64, true>::kOffTable <= kSmemLimit, "smem");
static_assert(Cfg<48, true>::kOffTable <= kSmemLimit, "smem");
static_assert(Cfg<64, false, false, false, true>::kOffTable <= kSmemLimit, "smem");
static_assert(Cfg<256, false, true>::kOffTable + 8 * (kMaxExperts + 1) <= kSmemLimit, "smem");
static_assert(Cfg<128, false, true>::kOffTable + 8 * (kMaxExperts + 1) <= kSmemLimit, "smem");
static_assert(Cfg<256, false, false, true>::kOffTable + 4 * (kMaxExperts + 1) <= kSmemLimit, "smem");
static_assert(Cfg<128, false, false, true>::kOffTable + 4 * (kMaxExperts + 1) <= kSmemLimit, "smem");

template <int BN, int MODE, bool PAIR = false, bool EPI = false>
int launch_kernel(const GemmArgs& args, const CUtensorMap& tA, const CUtensorMap& tB,
                  const CUtensorMap& tD, const CUtensorMap& tSA, const CUtensorMap& tSB, int grid,
                  int table_entries, cudaStream_t stream) {
  using C = CfgOf<BN, MODE, PAIR>;
  auto kern = fp8_gemm_kernel<BN, MODE, PAIR, EPI>;
  static std::atomic<uint64_t> attr_set{0};  // one bit per device
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemLimit)) != cudaSuccess) {
      cudaGetLastError();
      return FP8G_ERR_CUDA;
    }
    if constexpr (C::kRebalance) {
      // setmaxnreg.inc waits until the registers it asks for are free: the launch must hold
      // at least what the rebalanced warpgroups use, or the epilogue would never start.
      cudaFuncAttributes fa{};
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
        cudaGetLastError();
        return FP8G_ERR_CUDA;
      }
      if (fa.numRegs * C::kThreads < 128 * static_cast<int>(C::kRegsLow) +
                                         (C::kThreads - 128) * static_cast<int>(C::kRegsHigh))
        return FP8G_ERR_CUDA;
    }
    attr_set.fetch_or(bit);
  }
  const uint32_t smem = smem_bytes<BN, MODE == kDenseSmallM, PAIR, MODE == kKGrouped, MODE == kSwapAB>(table_entries);
  if constexpr (PAIR) {  // clusters of two CTAs (the grid is even)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tA, tB, tD, tSA, tSB, args) != cudaSuccess) {
      cudaGetLastError();
      return FP8G_ERR_CUDA;
    }
    return FP8G_OK;
  }
  if (args.ck > 1) {
    // cluster K split: clusters of ck CTAs (the grid is a multiple of ck), co-scheduled, so that
    // rank 0's wait for the other ranks' partials always ends
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(args.ck);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tA, tB, tD, tSA, tSB, args) != cudaSuccess) {
      cudaGetLastError();
      return FP8G_ERR_CUDA;
    }
    return FP8G_OK;
  }
  if (args.sk) {
    // stream-K: a CTA finishing a split tile waits for other CTAs' partials, so every CTA must
    // be resident at once -- a cooperative launch guarantees it (one CTA per SM, grid <= SMs)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tA, tB, tD, tSA, tSB, args) != cudaSuccess) {
      cudaGetLastError();
      return FP8G_ERR_CUDA;
    }
    return FP8G_OK;
  }
  // a programmatic dependent launch: the CTAs may start while the previous kernel on the stream
  // finishes (their prologue overlaps its tail) and wait for it before reading inputs
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tA, tB, tD, tSA, tSB, args) != cudaSuccess) {
    cudaGetLastError();
    return FP8G_ERR_CUDA;
  }
  return FP8G_OK;
}

// Stream-K workspace: one per (device, stream), allocated on the first call that needs it and
// kept for the life of the process.  Per stream, because launches on different streams may run
// at the same time; launches on one stream run in order and reuse it.  It holds one FP32
// partial-tile slot per SM (kSkSlotBytes: 128 x 128 columns x 2 column groups at most) and one
// flag per SM.
static_assert(kSkSlotBytes == static_cast<size_t>(BM) * 256 * 4, "stream-K slot size");
struct SkWorkspace {
  void* base = nullptr;
  size_t flag_offset = 0;
};
std::mutex g_sk_mutex;
std::map<std::pair<int, cudaStream_t>, SkWorkspace>* g_sk_ws = nullptr;

// The workspace of (device, stream), or false when there is none and it cannot be made now
// (allocation failed, or the stream is being captured into a graph: no allocation inside a
// capture -- the call then runs without the stream-K tail).
bool sk_workspace(int dev, int sm_count, cudaStream_t stream, float4** part, uint32_t** flags) {
  std::lock_guard<std::mutex> lock(g_sk_mutex);
  if (!g_sk_ws) g_sk_ws = new std::map<std::pair<int, cudaStream_t>, SkWorkspace>();
  SkWorkspace& w = (*g_sk_ws)[{dev, stream}];
  if (!w.base) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return false;
    }
    const size_t part_bytes = kSkSlotBytes * static_cast<size_t>(sm_count);
    const size_t flag_bytes = (static_cast<size_t>(sm_count) * 4 + 255) / 256 * 256;
    void* p = nullptr;
    if (cudaMalloc(&p, part_bytes + flag_bytes) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    w.base = p;
    w.flag_offset = part_bytes;
  }
  *part = static_cast<float4*>(w.base);
  *flags = reinterpret_cast<uint32_t*>(static_cast<char*>(w.base) + w.flag_offset);
  return true;
}

// FP8G_TEST_SKIP_STAGE=<n> (tests only, read on every call): the producer of every CTA leaves its
// stage n unfilled, so the issuer's wait for it runs out (see GemmArgs::test_skip_stage).
int env_test_skip_stage() {
  const char* e = std::getenv("FP8G_TEST_SKIP_STAGE");
  return e ? std::atoi(e) : -1;
}

// Raster band height (m-blocks).  Tiles run m-block fastest within a band of m-blocks and n-block
// by n-block, so the CTAs in flight share the band's A rows and a few B column blocks in L2.
//   Dense: when all of A fits well inside L2 (<= 48 MB) the band is all of M, so each B column
//   block is read from DRAM once with A staying resident (4096 x 8192 x 8192: 220 us against 226
//   with 16 m-blocks); otherwise 16 m-blocks (2048 rows), whose A slab stays resident while B
//   streams once per band.
//   Contiguous-grouped: 8 m-blocks.  A band spanning every expert keeps all experts' B column blocks
//   in flight at once (the grouped data gradient, 8576 x 7168 x 4096: 248 us with all 67 m-blocks,
//   226 us with 8 or 16; the MoE forward GEMM: 231 us with 8, 236 us with 16; again with the current
//   kernel: 220-221 us with 8, 224 with 4, 225 with 6, 230 with 10, 223 with 12, 221 with 16).
//   K-grouped: 16.
// FP8G_BAND_M overrides (read on every call).
int32_t band_rows(int32_t num_m, int64_t K, int mode) {
  if (const char* e = std::getenv("FP8G_BAND_M")) {
    const int v = std::atoi(e);
    if (v > 0) return v;
  }
  if (mode == kContiguous) return 8;
  if (mode != kDense) return kBandM;
  const int64_t a_bytes = static_cast<int64_t>(num_m) * BM * K;
  return a_bytes <= (int64_t{48} << 20) ? (num_m > 0 ? num_m : 1) : kBandM;
}

// FP8G_SWAP_AB=1 runs M <= 64 with swapped tiles (read on every call); otherwise the 64-wide small-M
// tiles.  Off by default: on 64 x 7168 x 7168 the swapped kernel took 21 us with its K blocks split
// over all SMs (28 us unsplit, on 56 SMs) against 19.7 us for the 64-wide tiles on 112 SMs (device
// times); the split's flag memset and cooperative launch add ~4 us more per call.  Both tile forms
// stream ~27 bytes per cycle per SM through TMA, so the larger weight share of a swapped stage
// (two thirds against one half) did not pay for the split.
bool env_swap_ab() {
  const char* e = std::getenv("FP8G_SWAP_AB");
  return e && e[0] == '1' && e[1] == 0;
}
// FP8G_CLUSTER_K=c (2 .. 8) forces the cluster K split with clusters of c CTAs where it applies,
// FP8G_CLUSTER_K=0 turns it off (read on every call); -1 when unset: the split is then chosen by
// cluster_k_auto.
int env_cluster_k() {
  const char* e = std::getenv("FP8G_CLUSTER_K");
  if (!e) return -1;
  if (e[0] == '0' && e[1] == 0) return 0;
  if (e[0] < '2' || e[0] > '8' || e[1] != 0) return -1;
  return e[0] - '0';
}

// The cluster K split by default: for dense block-scaled calls with few 256-wide tiles (at most half
// the SMs) and a long K (128 K blocks or more), the largest cluster of 8, 4 or 2 CTAs whose tiles
// fit on the SMs, that divides the K blocks and leaves each rank 16 or more.  Measured (device time):
// 128 x 1024 x 16384 41.7 -> 26.6 us, 128 x 2048 x 32768 80.9 -> 38.9, 512 x 1536 x 16384 43.0 ->
// 32.7; with 64 K blocks (256 x 2048 x 8192) it did not pay, nor for 64 rows or fewer (the small-M
// tiles, 64 x 4096 x 16384: 28.8 against 32.8 us).
int cluster_k_auto(int64_t tiles256, int64_t KB, int sm_count) {
  if (KB < 128 || tiles256 < 1 || 2 * tiles256 > sm_count) return 0;
  for (int c = 8; c >= 2; c /= 2)
    if (tiles256 * c <= sm_count && KB % c == 0 && KB / c >= 16) return c;
  return 0;
}

// FP8G_STREAMK=0 turns the stream-K tail off (read on every call).
bool env_streamk() {
  const char* e = std::getenv("FP8G_STREAMK");
  return !(e && e[0] == '0' && e[1] == 0);
}

thread_local int t_last_bn = 0, t_last_stages = 0, t_last_grid = 0, t_last_split = 0, t_last_swap = 0;
thread_local int t_last_ck = 0;

// FP8G_PAIR=1 runs 256-wide tiles as 256 x 256 CTA-pair tiles, FP8G_PAIR=2 as 256 x 128 pair
// tiles (four TMEM partial buffers per CTA).  Off by default: measured no faster than single-CTA
// 256-wide tiles (=1: within a few percent either way; =2: ~1.5x slower on 4096 x 8192 x 8192).
int env_pair() {
  const char* e = std::getenv("FP8G_PAIR");
  return (e && (e[0] == '1' || e[0] == '2') && e[1] == 0) ? e[0] - '0' : 0;
}

// FP8G_BLOCK_N (48, 64, 128, 160, 192 or 256) forces the tile width; read on every call (48: decode
// shapes only).  160 and 192
// are only taken this way: measured slower than 256 on the large shapes (4096 x 8192 x 8192: 361 and
// 288 us against 212).  Per K block a narrower tile still needs four tcgen05.mma, and one issuing
// thread took ~620 cycles for the four N = 160 MMAs and their commit against ~325 cycles of MMA
// work (a second issuer measured the same), so those tiles are issue-bound.
int env_block_n() {
  const char* e = std::getenv("FP8G_BLOCK_N");
  const int x = e ? std::atoi(e) : 0;
  return (x == 48 || x == 64 || x == 128 || x == 160 || x == 192 || x == 256) ? x : 0;
}

// Pick BN: fewest (waves x per-tile cost), the per-tile cost growing with BN plus a fixed
// promotion/epilogue overhead.  Small-M shapes get narrow tiles so that every SM streams B.
// The epilogue-scaled variant has no 64-wide tiles (min_bn 128).
int choose_block_n(int64_t m_blocks, int64_t N, int sms, int min_bn = 64) {
  if (int v = env_block_n()) return v < min_bn ? min_bn : v;
  int best = 256;
  double best_cost = 1e300;
  for (int bn : {256, 128, 64}) {
    if (bn < min_bn) continue;
    const int64_t tiles = m_blocks * ((N + bn - 1) / bn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double cost = static_cast<double>(waves) * (bn + 64);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

struct Operands {
  const void* A;
  int64_t lda;
  const float* sA;
  int64_t ld_sa;
  const void* B;
  int64_t ldb;
  const float* sB;
  void* D;
  int64_t ldd;
  int64_t rows, N, K, E, cap;
  const int32_t* groups;
  int32_t sa_step = 0, sb_step = 0;  // epilogue-scaled variant only
  uint32_t idesc_fmt = 0;             // operand formats (A e5m2: 1 << 7)
  int64_t ld_sb = 0;                  // kKGrouped: B scales [K blocks][ld_sb]
};

// EPI: the epilogue-scaled variant (per-tensor / per-token / per-channel scales)
template <int MODE, bool EPI = false>
int run_gemm(const Operands& o, cudaStream_t stream, bool no_alloc = false) {
  DeviceInfo* dev = nullptr;
  int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  if (o.rows == 0) return FP8G_OK;

  const int64_t m_blocks = (MODE == kMasked)     ? o.E * ((o.cap + BM - 1) / BM)
                           : (MODE == kKGrouped) ? o.E * ((o.rows + BM - 1) / BM)
                                                 : (o.rows + BM - 1) / BM;
  int bn = choose_block_n(m_blocks, o.N, dev->sm_count, (EPI || MODE == kKGrouped) ? 128 : 64);
  if ((EPI || MODE == kKGrouped) && (bn == 192 || bn == 160)) bn = 256;  // those forms: 128 and 256 wide
  if (bn == 160 && MODE != kDense && o.E > kMaxExperts160) bn = 256;    // group table too large
  // decode shapes (at most 64 rows of A, block-scaled dense): with FP8G_SWAP_AB=1 (and no tile width
  // forced by FP8G_BLOCK_N) swapped tiles, weight rows on the MMA's M; else 64-wide tiles in the
  // small-M variant (64-row A boxes)
  const bool swap = MODE == kDense && !EPI && o.rows <= 64 && env_block_n() == 0 && env_swap_ab();
  if (swap) bn = 64;
  // cluster K split: 256-wide single-CTA tiles, each computed by a cluster of CTAs (forced with
  // FP8G_CLUSTER_K, else chosen for few tiles with a long K, above the small-M shapes)
  int ck_req = 0;
  if (MODE == kDense && !EPI && !swap && !no_alloc) {
    const int ce = env_cluster_k();
    const int64_t tiles256 = ((o.rows + BM - 1) / BM) * ((o.N + 255) / 256);
    ck_req = ce >= 0 ? ce : (o.rows > 64 && env_block_n() == 0 && env_pair() == 0 ? cluster_k_auto(tiles256, o.K / BK, dev->sm_count) : 0);
  }
  if (ck_req > 1) bn = 256;
  // Small-M tiles are 64 wide, or 48 with FP8G_BLOCK_N=48 (other shapes and forms have no 48-wide
  // tiles).  On 64 x 7168 x 7168 the 150 48-wide tiles measured no faster than the 112 64-wide ones
  // (25.2 us either way): each CTA still walks all 56 K blocks at the same ~590 cycles a block, and
  // that serial loop, not the number of SMs streaming, sets the time.
  const bool small_ok = MODE == kDense && !EPI && !swap && o.rows <= 64;
  if (!small_ok && bn == 48) bn = 64;
  const bool small_m = small_ok && (bn == 64 || bn == 48);
  // 256-wide tiles run as CTA pairs unless there are too few rows: 256 x 256 pair tiles
  // (FP8G_PAIR=1) or 256 x 128 (FP8G_PAIR=2); the epilogue-scaled variant has single-CTA tiles
  const int pmode = (EPI || MODE == kKGrouped) ? 0 : env_pair();
  const bool pair = bn == 256 && pmode != 0 && ck_req <= 1 &&
                    (MODE != kDense || (o.rows + BM - 1) / BM >= 2) && dev->sm_count >= 2;
  if (pair && pmode == 2) bn = 128;

  GemmArgs a{};
  a.rows = static_cast<int32_t>(o.rows);
  a.N = static_cast<int32_t>(o.N);
  a.KB = static_cast<int32_t>(o.K / BK);
  a.NBs = static_cast<int32_t>((o.N + 127) / 128);
  a.E = static_cast<int32_t>(o.E);
  a.cap = static_cast<int32_t>(o.cap);
  a.num_m = static_cast<int32_t>((o.rows + BM - 1) / BM);
  a.num_n = static_cast<int32_t>((o.N + bn - 1) / bn);
  a.num_tiles = a.num_m * a.num_n;
  a.sA = o.sA;
  a.ld_sa = o.ld_sa;
  a.sB = o.sB;
  a.D = static_cast<__nv_bfloat16*>(o.D);
  a.ldd = o.ldd;
  a.groups = o.groups;
  a.status = dev->status;
  a.budget = wait_budget_cycles();
  a.sa_step = o.sa_step;
  a.sb_step = o.sb_step;
  a.idesc_fmt = o.idesc_fmt;
  a.ld_sb = o.ld_sb;
  a.test_skip_stage = env_test_skip_stage();
  a.band_m = band_rows(a.num_m, o.K, MODE == kDenseSmallM ? kDense : MODE);
  if (MODE == kKGrouped) a.num_tiles = static_cast<int32_t>(o.E) * a.num_m * a.num_n;
  if (swap) {
    // D^T = B A^T: rows are the weight rows, columns the tokens; one 128-row weight slab a tile.
    // sA (token scales [K/128][ld_sa]) and sB (weight block scales [N/128][K/128]) keep their
    // meaning; the A and B operand formats trade places in the instruction descriptor.
    a.rows = static_cast<int32_t>(o.N);
    a.N = static_cast<int32_t>(o.rows);
    a.num_m = static_cast<int32_t>((o.N + BM - 1) / BM);
    a.num_n = 1;
    a.num_tiles = a.num_m;
    a.band_m = band_rows(a.num_m, o.K, kDense);
    a.idesc_fmt = (((o.idesc_fmt >> 7) & 7u) << 10) | (((o.idesc_fmt >> 10) & 7u) << 7);
  }

  // K blocks per stage of the variant launched below (its Cfg::kKPS)
  const uint32_t kps = small_m ? Cfg<64, true>::kKPS : (swap ? Cfg<64, false, false, false, true>::kKPS : 1u);
  CUtensorMap tA, tB, tD;
  if (swap) {
    // the MMA's A: the weights as [K/128][N][128], a box of kps K blocks of a 128-row slab
    const uint64_t dims[3] = {BK, static_cast<uint64_t>(o.N), static_cast<uint64_t>(o.K / BK)};
    const uint64_t strides[2] = {static_cast<uint64_t>(o.ldb), BK};
    const uint32_t box[3] = {BK, static_cast<uint32_t>(BM), kps};
    if ((st = encode_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, o.B, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != FP8G_OK)
      return st;
  } else {
    // A as [K/128][rows][128]: a box is kps K blocks of the tile's rows
    const uint64_t dims[3] = {BK, static_cast<uint64_t>(o.rows), static_cast<uint64_t>(o.K / BK)};
    const uint64_t strides[2] = {static_cast<uint64_t>(o.lda), BK};
    const uint32_t box[3] = {BK, small_m ? 64u : static_cast<uint32_t>(BM), kps};
    if ((st = encode_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, o.A, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != FP8G_OK)
      return st;
  }
  if (swap) {
    // the MMA's B: the activations as [1][K/128][M][128], a box of kps K blocks of 64 token rows
    // (rows past M read as zero)
    const uint64_t dims[4] = {BK, static_cast<uint64_t>(o.rows), static_cast<uint64_t>(o.K / BK), 1};
    const uint64_t strides[3] = {static_cast<uint64_t>(o.lda), BK, static_cast<uint64_t>(o.lda * o.rows)};
    const uint32_t box[4] = {BK, 64u, kps, 1};
    if ((st = encode_tmap(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, o.A, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != FP8G_OK)
      return st;
  } else {
    // B as [E][K/128][N][128]
    const uint64_t dims[4] = {BK, static_cast<uint64_t>(o.N), static_cast<uint64_t>(o.K / BK),
                              static_cast<uint64_t>(MODE == kKGrouped ? 1 : o.E)};
    const uint64_t strides[3] = {static_cast<uint64_t>(o.ldb), BK, static_cast<uint64_t>(o.ldb * o.N)};
    const uint32_t box[4] = {BK, static_cast<uint32_t>(pair ? bn / 2 : bn), kps, 1};
    if ((st = encode_tmap(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, o.B, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != FP8G_OK)
      return st;
  }
  // Scales staged per stage (block-scaled forms): sA as [K/128][rows] fp32 with row stride ld_sa,
  // a box being the 128 A-row scales of a tile for kps K blocks (rows past the matrix read as
  // zero); K-grouped: the per-column B scales as [T/128][N] (row stride ld_sb), a box of BN.
  // The epilogue-scaled variant reads its scales directly; its maps are unused placeholders.
  CUtensorMap tSA = tA, tSB = tA;
  if (!EPI) {
    const uint64_t dims[2] = {static_cast<uint64_t>(o.rows), static_cast<uint64_t>(o.K / BK)};
    const uint64_t strides[1] = {static_cast<uint64_t>(o.ld_sa) * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(BM), kps};
    if ((st = encode_tmap(&tSA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, o.sA, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != FP8G_OK)
      return st;
  }
  if (MODE == kKGrouped) {
    const uint64_t dims[2] = {static_cast<uint64_t>(o.N), static_cast<uint64_t>(o.K / BK)};
    const uint64_t strides[1] = {static_cast<uint64_t>(o.ld_sb) * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(bn), 1};
    if ((st = encode_tmap(&tSB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, o.sB, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) != FP8G_OK)
      return st;
  }
  {
    // D: [rows, N] (K-grouped: one [rows, N] matrix per expert, stacked)
    const uint64_t d_rows = static_cast<uint64_t>(MODE == kKGrouped ? o.E * o.rows : o.rows);
    const uint64_t dims[2] = {static_cast<uint64_t>(o.N), d_rows};
    const uint64_t strides[1] = {static_cast<uint64_t>(o.ldd * 2)};
    const uint32_t box[2] = {32, 32};
    if ((st = encode_tmap(&tD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.D, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_64B)) != FP8G_OK)
      return st;
  }

  int64_t tiles_upper = (MODE == kMasked) ? m_blocks * a.num_n : static_cast<int64_t>(a.num_tiles);
  int grid = static_cast<int>(std::min<int64_t>(std::max<int64_t>(tiles_upper, 1), dev->sm_count));
  // stream-K tail for single-CTA tiles of width >= 128 (one K part, one MMA issuer) when the
  // tiles do not fill whole rounds of the grid (masked: the count is only known on the device)
  a.sk = 0;
  a.sk_min_units = 8;
  // a split tile costs its CTAs ~8-9 us (FP32 partial written, read back and added, and one more
  // tile hand-off), about 20 K blocks of MMA time: split only when that gains clearly more
  a.sk_min_gain = 24;
  // (the same split rule as make_work on the device; the masked tile count is only known there)
  auto tail_splits = [&](int64_t T) {
    const int64_t G = dev->sm_count, KB = a.KB;
    const int64_t U = (T - T / G * G) * KB;
    int64_t u = (U + G - 1) / G;
    const int64_t umin = a.sk_min_units < KB ? a.sk_min_units : KB;
    if (u < umin) u = umin;
    return U > 0 && KB - u >= a.sk_min_gain;
  };
  // (160-wide tiles have two MMA issuers, which take whole tiles; swapped tiles split too: their
  // N / 128 weight slabs are fewer than the SMs)
  // cluster K split: every tile gets a cluster of ck CTAs when they all fit on the SMs at once and
  // ck divides the K blocks, at least two a rank (the clusters wait only within themselves)
  a.ck = 0;
  if (ck_req > 1 && !pair && static_cast<int64_t>(a.num_tiles) * ck_req <= dev->sm_count && a.KB % ck_req == 0 &&
      a.KB >= 2 * ck_req) {
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    if (sk_workspace(dev_id, dev->sm_count, stream, &a.ws_part, &a.ws_flag)) {
      a.ck = ck_req;
      grid = a.num_tiles * ck_req;
    }
  }
  if (a.ck <= 1 && MODE != kKGrouped && !pair && !small_m && (swap || (bn >= 128 && bn != 160)) && env_streamk() &&
      (MODE == kMasked || tail_splits(a.num_tiles))) {
    int dev_id = 0;
    cudaGetDevice(&dev_id);
    bool have_ws = false;
    if (no_alloc) {  // the fixed scratch (the caller has checked that it holds every SM's slot)
      void* p = noalloc_scratch(dev_id);
      if (!p) return FP8G_ERR_CUDA;
      a.ws_part = static_cast<float4*>(p);
      a.ws_flag = reinterpret_cast<uint32_t*>(static_cast<char*>(p) + kSkSlotBytes * kNoAllocSlots);
      have_ws = true;
    } else {
      have_ws = sk_workspace(dev_id, dev->sm_count, stream, &a.ws_part, &a.ws_flag);
    }
    if (have_ws) {
      if (cudaMemsetAsync(a.ws_flag, 0, static_cast<size_t>(dev->sm_count) * 4, stream) != cudaSuccess) {
        cudaGetLastError();
        return FP8G_ERR_CUDA;
      }
      a.sk = 1;
      grid = dev->sm_count;  // every SM takes a share of the tail
    }
  }
  int table_entries = (MODE == kDense) ? 0 : static_cast<int>(o.E + 1);
  if (pair) {
    // pair tiles: dense ceil(num_m/2) x num_n; grouped at most (m-blocks + experts)/2 x num_n
    if (MODE == kDense) a.num_tiles = ((a.num_m + 1) / 2) * a.num_n;
    const int64_t pair_upper = (MODE == kDense) ? a.num_tiles : ((m_blocks + o.E + 1) / 2) * a.num_n;
    grid = 2 * static_cast<int>(std::min<int64_t>(std::max<int64_t>(pair_upper, 1), dev->sm_count / 2));
    if (MODE != kDense) table_entries = 2 * static_cast<int>(o.E + 1);
  }

  t_last_bn = bn;
  t_last_grid = grid;
  t_last_split = a.sk;
  t_last_ck = a.ck;
  t_last_swap = swap ? 1 : 0;
  if constexpr (MODE == kKGrouped) {
    if (bn == 256) {
      t_last_stages = Cfg<256, false, false, true>::kStages;
      return launch_kernel<256, kKGrouped>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
    }
    t_last_stages = Cfg<128, false, false, true>::kStages;
    return launch_kernel<128, kKGrouped>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
  } else if constexpr (EPI) {
    if (bn == 256) {
      t_last_stages = Cfg<256>::kStages;
      return launch_kernel<256, MODE, false, true>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
    }
    t_last_stages = Cfg<128>::kStages;
    return launch_kernel<128, MODE, false, true>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
  } else {
    if constexpr (MODE == kDense) {
      if (swap) {
        t_last_stages = Cfg<64, false, false, false, true>::kStages;
        return launch_kernel<64, kSwapAB>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
      }
    }
    switch (bn) {
      case 256:
        if (pair) {
          t_last_stages = Cfg<256, false, true>::kStages;
          return launch_kernel<256, (MODE == kDenseSmallM ? kDense : MODE), true>(a, tA, tB, tD, tSA, tSB, grid,
                                                                                 table_entries, stream);
        }
        t_last_stages = Cfg<256>::kStages;
        return launch_kernel<256, MODE>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
      case 192:
        t_last_stages = Cfg<192>::kStages;
        return launch_kernel<192, MODE>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
      case 160:
        t_last_stages = Cfg<160>::kStages;
        return launch_kernel<160, MODE>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
      case 128:
        if (pair) {
          t_last_stages = Cfg<128, false, true>::kStages;
          return launch_kernel<128, (MODE == kDenseSmallM ? kDense : MODE), true>(a, tA, tB, tD, tSA, tSB, grid,
                                                                                 table_entries, stream);
        }
        t_last_stages = Cfg<128>::kStages;
        return launch_kernel<128, MODE>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
      case 48:
        if constexpr (MODE == kDense) {
          t_last_stages = Cfg<48, true>::kStages;
          return launch_kernel<48, kDenseSmallM>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
        }
        return FP8G_ERR_INVALID_ARG;
      default:
        if constexpr (MODE == kDense) {
          if (small_m) {
            t_last_stages = Cfg<64, true>::kStages;
            return launch_kernel<64, kDenseSmallM>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
          }
        }
        t_last_stages = Cfg<64>::kStages;
        return launch_kernel<64, MODE>(a, tA, tB, tD, tSA, tSB, grid, table_entries, stream);
    }
  }
}

constexpr int64_t kMaxI32 = 0x7FFFFFFF;

}  // namespace
}  // namespace fp8g

using namespace fp8g;

extern "C" int fp8_gemm_nt(const void* A, int64_t lda, const float* sA, int64_t ld_sa,
                           const void* B, int64_t ldb, const float* sB, void* D, int64_t ldd,
                           int64_t M, int64_t N, int64_t K, void* stream) {
  if (M < 0 || M > kMaxI32 || N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 ||
      K > kMaxI32)
    return FP8G_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldd < N || ld_sa < M) return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;  // nothing to do; the pointers of empty tensors may be null
  if (!A || !sA || !B || !sB || !D) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      lda % 16 != 0 || ldb % 16 != 0 || ldd % 8 != 0 || ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, lda, sA, ld_sa, B, ldb, sB, D, ldd, M, N, K, 1, 0, nullptr};
  return run_gemm<kDense>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_gemm_nt_noalloc(const void* A, int64_t lda, const float* sA, int64_t ld_sa,
                                   const void* B, int64_t ldb, const float* sB, void* D,
                                   int64_t ldd, int64_t M, int64_t N, int64_t K, void* stream) {
  // the argument rules of fp8_gemm_nt
  if (M < 0 || M > kMaxI32 || N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 ||
      K > kMaxI32)
    return FP8G_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldd < N || ld_sa < M) return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;
  if (!A || !sA || !B || !sB || !D) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      lda % 16 != 0 || ldb % 16 != 0 || ldd % 8 != 0 || ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  // the fixed scratch holds kNoAllocSlots SMs' slots: a larger device is out of its range
  DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  if (dev->sm_count > kNoAllocSlots) return FP8G_ERR_INVALID_ARG;
  Operands o{A, lda, sA, ld_sa, B, ldb, sB, D, ldd, M, N, K, 1, 0, nullptr};
  return run_gemm<kDense>(o, static_cast<cudaStream_t>(stream), true);
}

extern "C" int fp8_grouped_gemm_contiguous(const void* A, const float* sA, int64_t ld_sa,
                                           const void* B, const float* sB, void* D,
                                           const int32_t* group_offsets, int32_t E,
                                           int64_t M_total, int64_t N, int64_t K, void* stream) {
  if (E < 1 || E > kMaxExperts || M_total < 0 || M_total > kMaxI32 || M_total % 128 != 0 ||
      N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 || K > kMaxI32 ||
      ld_sa < M_total)
    return FP8G_ERR_INVALID_ARG;
  if (M_total == 0) return FP8G_OK;
  if (!A || !sA || !B || !sB || !D || !group_offsets) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      (reinterpret_cast<uintptr_t>(group_offsets) & 3u) || ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, K, sA, ld_sa, B, K, sB, D, N, M_total, N, K, E, 0, group_offsets};
  return run_gemm<kContiguous>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_grouped_gemm_masked(const void* A, const float* sA, int64_t ld_sa,
                                       const void* B, const float* sB, void* D,
                                       const int32_t* masked_m, int32_t E, int64_t cap, int64_t N,
                                       int64_t K, void* stream) {
  if (E < 1 || E > kMaxExperts || cap < 0 || cap % 16 != 0 || static_cast<int64_t>(E) * cap > kMaxI32 ||
      N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 || K > kMaxI32 ||
      ld_sa < static_cast<int64_t>(E) * cap)
    return FP8G_ERR_INVALID_ARG;
  if (cap == 0) return FP8G_OK;
  if (!A || !sA || !B || !sB || !D || !masked_m) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      (reinterpret_cast<uintptr_t>(masked_m) & 3u) || ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, K, sA, ld_sa, B, K, sB, D, N, static_cast<int64_t>(E) * cap, N, K, E, cap, masked_m};
  return run_gemm<kMasked>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_gemm_nt_dgrad(const void* A, int64_t lda, const float* sA, int64_t ld_sa,
                                 const void* B, int64_t ldb, const float* sB, void* D, int64_t ldd,
                                 int64_t M, int64_t N, int64_t K, void* stream) {
  // the argument rules of fp8_gemm_nt; A holds e5m2 codes
  if (M < 0 || M > kMaxI32 || N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 ||
      K > kMaxI32)
    return FP8G_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldd < N || ld_sa < M) return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;
  if (!A || !sA || !B || !sB || !D) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      lda % 16 != 0 || ldb % 16 != 0 || ldd % 8 != 0 || ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, lda, sA, ld_sa, B, ldb, sB, D, ldd, M, N, K, 1, 0, nullptr};
  o.idesc_fmt = 1u << 7;  // A: e5m2
  return run_gemm<kDense>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_grouped_gemm_contiguous_dgrad(const void* A, const float* sA, int64_t ld_sa,
                                                 const void* B, const float* sB, void* D,
                                                 const int32_t* group_offsets, int32_t E,
                                                 int64_t M_total, int64_t N, int64_t K, void* stream) {
  // the argument rules of fp8_grouped_gemm_contiguous; A holds e5m2 codes
  if (E < 1 || E > kMaxExperts || M_total < 0 || M_total > kMaxI32 || M_total % 128 != 0 ||
      N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 || K > kMaxI32 ||
      ld_sa < M_total)
    return FP8G_ERR_INVALID_ARG;
  if (M_total == 0) return FP8G_OK;
  if (!A || !sA || !B || !sB || !D || !group_offsets) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      (reinterpret_cast<uintptr_t>(group_offsets) & 3u) || ld_sa % 4 != 0)
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, K, sA, ld_sa, B, K, sB, D, N, M_total, N, K, E, 0, group_offsets};
  o.idesc_fmt = 1u << 7;  // A: e5m2
  return run_gemm<kContiguous>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_grouped_gemm_wgrad(const void* A, int64_t lda, const float* sA, int64_t ld_sa,
                                      const void* B, int64_t ldb, const float* sB, int64_t ld_sb,
                                      void* D, const int32_t* offsets, int32_t E, int64_t M, int64_t N,
                                      int64_t T, void* stream) {
  if (E < 1 || E > kMaxExperts || M < 0 || M % 16 != 0 || static_cast<int64_t>(E) * M > kMaxI32 ||
      N <= 0 || N > kMaxI32 || N % 16 != 0 || T <= 0 || T % 128 != 0 || T > kMaxI32 || lda < T ||
      ldb < T || ld_sa < M || ld_sb < N)
    return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;
  if (!A || !sA || !B || !sB || !D || !offsets) return FP8G_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(sA) || !aligned16(B) || !aligned16(sB) || !aligned16(D) ||
      lda % 16 != 0 || ldb % 16 != 0 || ld_sa % 4 != 0 || ld_sb % 4 != 0 ||
      (reinterpret_cast<uintptr_t>(offsets) & 3u))
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, lda, sA, ld_sa, B, ldb, sB, D, N, M, N, T, E, 0, offsets};
  o.idesc_fmt = 1u << 7;  // A (the output gradient): e5m2
  o.ld_sb = ld_sb;
  return run_gemm<kKGrouped>(o, static_cast<cudaStream_t>(stream));
}

// Epilogue-scaled forms: the scale arguments are checked here, the rest as in the block-scaled
// entry points.  sA: 4-byte aligned; sB: 16-byte aligned when it has one scale per column
// (read as float4), else 4-byte aligned.
namespace {
int check_epi_scales(const float* sA, int32_t sa_per_row, const float* sB, int32_t sb_per_col) {
  if ((sa_per_row != 0 && sa_per_row != 1) || (sb_per_col != 0 && sb_per_col != 1)) return FP8G_ERR_INVALID_ARG;
  if (!sA || !sB) return FP8G_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(sA) & 3u) ||
      (reinterpret_cast<uintptr_t>(sB) & (sb_per_col ? 15u : 3u)))
    return FP8G_ERR_ALIGNMENT;
  return FP8G_OK;
}
}  // namespace

extern "C" int fp8_gemm_nt_scaled(const void* A, int64_t lda, const float* sA, int32_t sa_per_row,
                                  const void* B, int64_t ldb, const float* sB, int32_t sb_per_col,
                                  void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, void* stream) {
  if (M < 0 || M > kMaxI32 || N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 ||
      K > kMaxI32 || lda < K || ldb < K || ldd < N)
    return FP8G_ERR_INVALID_ARG;
  if (sa_per_row != 0 && sa_per_row != 1) return FP8G_ERR_INVALID_ARG;
  if (sb_per_col != 0 && sb_per_col != 1) return FP8G_ERR_INVALID_ARG;
  if (M == 0) return FP8G_OK;
  if (!A || !B || !D) return FP8G_ERR_INVALID_ARG;
  if (int st = check_epi_scales(sA, sa_per_row, sB, sb_per_col)) return st;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || lda % 16 != 0 || ldb % 16 != 0 || ldd % 8 != 0)
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, lda, sA, 0, B, ldb, sB, D, ldd, M, N, K, 1, 0, nullptr, sa_per_row, sb_per_col};
  return run_gemm<kDense, true>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_grouped_gemm_contiguous_scaled(const void* A, const float* sA, int32_t sa_per_row,
                                                  const void* B, const float* sB, int32_t sb_per_col,
                                                  void* D, const int32_t* group_offsets, int32_t E,
                                                  int64_t M_total, int64_t N, int64_t K, void* stream) {
  if (E < 1 || E > kMaxExperts || M_total < 0 || M_total > kMaxI32 || M_total % 128 != 0 ||
      N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 || K > kMaxI32)
    return FP8G_ERR_INVALID_ARG;
  if (sa_per_row != 0 && sa_per_row != 1) return FP8G_ERR_INVALID_ARG;
  if (sb_per_col != 0 && sb_per_col != 1) return FP8G_ERR_INVALID_ARG;
  if (M_total == 0) return FP8G_OK;
  if (!A || !B || !D || !group_offsets) return FP8G_ERR_INVALID_ARG;
  if (int st = check_epi_scales(sA, sa_per_row, sB, sb_per_col)) return st;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (reinterpret_cast<uintptr_t>(group_offsets) & 3u))
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, K, sA, 0, B, K, sB, D, N, M_total, N, K, E, 0, group_offsets, sa_per_row, sb_per_col};
  return run_gemm<kContiguous, true>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_grouped_gemm_masked_scaled(const void* A, const float* sA, int32_t sa_per_row,
                                              const void* B, const float* sB, int32_t sb_per_col,
                                              void* D, const int32_t* masked_m, int32_t E, int64_t cap,
                                              int64_t N, int64_t K, void* stream) {
  if (E < 1 || E > kMaxExperts || cap < 0 || cap % 16 != 0 || static_cast<int64_t>(E) * cap > kMaxI32 ||
      N <= 0 || N > kMaxI32 || N % 16 != 0 || K <= 0 || K % 128 != 0 || K > kMaxI32)
    return FP8G_ERR_INVALID_ARG;
  if (sa_per_row != 0 && sa_per_row != 1) return FP8G_ERR_INVALID_ARG;
  if (sb_per_col != 0 && sb_per_col != 1) return FP8G_ERR_INVALID_ARG;
  if (cap == 0) return FP8G_OK;
  if (!A || !B || !D || !masked_m) return FP8G_ERR_INVALID_ARG;
  if (int st = check_epi_scales(sA, sa_per_row, sB, sb_per_col)) return st;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (reinterpret_cast<uintptr_t>(masked_m) & 3u))
    return FP8G_ERR_ALIGNMENT;
  Operands o{A, K, sA, 0, B, K, sB, D, N, static_cast<int64_t>(E) * cap, N, K, E, cap, masked_m,
             sa_per_row, sb_per_col};
  return run_gemm<kMasked, true>(o, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8g_selftest_bounded_waits(int64_t budget_cycles, uint32_t* out, void* stream) {
  if (budget_cycles <= 0 || budget_cycles > (int64_t{1} << 40) || !out) return FP8G_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 3u) return FP8G_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != FP8G_OK) return st;
  GemmArgs a{};
  a.status = dev->status;
  a.budget = budget_cycles;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(a, out);
  return cudaGetLastError() == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA;
}

extern "C" int fp8g_last_split(int* split) {
  if (!split) return FP8G_ERR_INVALID_ARG;
  *split = t_last_split;
  return FP8G_OK;
}

extern "C" int fp8g_last_swap_ab(int* swapped) {
  if (!swapped) return FP8G_ERR_INVALID_ARG;
  *swapped = t_last_swap;
  return FP8G_OK;
}

extern "C" int fp8g_last_cluster_k(int* ck) {
  if (!ck) return FP8G_ERR_INVALID_ARG;
  *ck = t_last_ck;
  return FP8G_OK;
}

extern "C" int fp8g_last_config(int* block_n, int* stages, int* grid) {
  if (!block_n || !stages || !grid) return FP8G_ERR_INVALID_ARG;
  *block_n = t_last_bn;
  *stages = t_last_stages;
  *grid = t_last_grid;
  return FP8G_OK;
}
