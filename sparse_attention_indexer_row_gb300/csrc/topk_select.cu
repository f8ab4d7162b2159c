// Batched row-wise top-k for a sparse-attention indexer, GB300 (sm_103a).
//
// The selector streams every score of a row exactly once, in blocks visited in
// a seeded shuffled order, and asks each element one question: does it beat
// the row's threshold?  Survivors go to a small shared-memory tray; when the
// tray passes its high-water mark a bitonic sort runs on the tray only, keeps
// the best k and raises the threshold to the k-th of them; the threshold never
// falls.  (The Secret GPU Kernel Behind DeepSeek V4.1 Flash, video transcript
// 3:18-4:20; the shuffle 3:30 and 4:55-5:10; the 32-bit survivor mask
// 5:10-5:22; the split-row leader merge 5:33-5:45.)
//
// GB300 mapping:
//  * The shuffle runs over visiting units of eight consecutive 1024-element
//    blocks (32 KB), each moved by one cp.async.bulk copy into one stage of a
//    shared-memory ring.  On GB300 a ring fed with 4 KB copies in shuffled
//    order streams well under half of HBM bandwidth, while shuffled 32 KB
//    copies stream above 90% of it.  The order is still drawn from Philox
//    without looking at the scores, so no input can make it slow; the
//    survivor bound counts units instead of blocks.
//  * Work is cut into pieces (the units of one row that one CTA owns).
//    Inside a CTA three kinds of warps run side by side with no CTA-wide
//    barrier after set-up:
//      - the producer warp walks the CTA's plan, draws each piece's visiting
//        order, publishes a descriptor per piece and per stage and issues
//        the copies;
//      - filter warps test every element against the piece's threshold and
//        append survivors to the piece's inbox;
//      - selector warps set each piece's starting threshold as soon as its
//        first unit has landed (warm start: every selector warp finds, by
//        bisection over key bits, a key that at least ceil(k/8) of its 1024
//        elements of that unit reach, and the smallest of the eight keys is
//        reached by at least k elements of the piece), drain the inbox into
//        the tray, raise the threshold (histogram select + prune), run the
//        bitonic tray sort when the tray passes its mark, and finish each
//        piece.
//    Pieces alternate between two inboxes, so the selectors finish piece j
//    (final sort, output or split-row merge) while the filters already
//    stream piece j+1; the filters wait only before piece j+2.
//  * Two plans.  Short batches of full-length rows: a persistent grid of one
//    CTA per SM, each owning an equal share of the batch's units laid end to
//    end; rows that straddle a share boundary are split.  Otherwise: (row,
//    segment) items dealt round-robin to a persistent grid.
//  * Every element becomes the 64-bit word (order key << 32) | ~index.  The
//    order key is the usual monotone map of float bits, so word order is value
//    order with ties broken towards the smaller index, and one 64-bit compare
//    decides every question exactly.  (The packed 64-bit words of DeepSeek
//    V4.1 Flash, kernelbench model page, entry "Single-launch CUDA bitonic
//    selection"; the ~index half gives the smaller-index tie rule.)
//  * The per-element test first runs as one float compare that can only let
//    too much through (it passes NaN and values equal to the threshold's),
//    giving each lane a 32-bit candidate mask; a lane walks only its own set
//    bits for the exact word test.  Survivors are compacted with a warp
//    prefix of per-lane counts (ballots and __popc); one shared-memory
//    atomicAdd per warp and stage reserves inbox space.  An empty inbox slot
//    holds the word 0, which no element packs to, so the selectors can tell a
//    reserved slot whose word has not landed yet.
//  * Every 512 new tray words a byte-wise histogram select over kept + tray
//    finds a word prefix T with at least k words at or above it; tray words
//    below T can never reach the best k and are dropped, and the threshold
//    rises to T.  When the tray passes its 2048-word mark, and at the end of
//    a piece, the survivors are sorted by a bitonic network (up to three
//    strides per barrier round) and merged into the kept list: the
//    element-wise max of the kept list against the reversed sorted words is a
//    bitonic sequence holding the best k' of both (k' = k rounded up to a
//    power of two), and a bitonic merge sorts it; the threshold becomes the
//    k-th kept word.
//  * A split row's CTAs share the best threshold any of them has reached
//    through a 64-bit atomicMax word per row.  Each publishes its sorted local
//    top-k to the workspace, fences, and takes a ticket; the CTA that draws the
//    last ticket merges all lists (a tree of parallel pairwise merges in its
//    shared memory) and writes the row (the atomic-ticket last-CTA combine of
//    DeepSeek V4.1 Flash, kernelbench model page, entry on the split-KV paged
//    decode), then resets the ticket and threshold word for the next call.
//  * No kernel ever traps or waits without a bound: bad lengths and NaNs set
//    workspace status bits, and every wait (mbarrier, inbox room, inbox slot,
//    piece hand-over) gives up after a fixed number of polls, setting a status
//    bit; after one wait has given up the others poll once and the CTA drains.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "device_util.cuh"
#include "topk_select.h"

namespace topk {
namespace {

constexpr int kBlock = 1024;                 // elements per block ("blocks of 1,024")
constexpr int kUnitBlocks = 8;               // blocks per visiting unit
constexpr int kUnit = kBlock * kUnitBlocks;  // elements per unit = per ring stage (32 KB)
constexpr int kPermChunk = 256;              // units shuffled together (2M elements)
constexpr int kTrayMark = 2048;              // tray words that trigger the tray sort
constexpr int kPruneStep = 512;              // new tray words that trigger a prune
constexpr int kSelectSlack = 256;            // extra words a pruned tray may keep
constexpr int kWarmUnits = 4;                // units a warm start reads at most (see warm_units)
constexpr int kWarmUnitsSmallK = 3;          // ... when each selector warp needs <= 64 (k <= 512)
// (k <= 512 runs a five-stage ring: the producer lands the three warm-start
// units of a piece while the filters hold its first one and keeps two more
// copies in flight; above, the four warm-start units of a long row fill the
// four-stage ring)
static_assert(kWarmUnits <= 4 && kWarmUnitsSmallK <= kWarmUnits,
              "warm-start units fit in the smallest ring");
// Speculative start: a piece with a full warm-start sample may start from a
// threshold those units only make likely (about 3.6 k words of the row above
// it).  It is taken when they hold at least 2.5 k * sample / row length
// elements at or above it, at most kSpecMaxNeed (so: long rows).
constexpr uint32_t kSpecMaxNeed = 256;
constexpr int kRescanChunk = 2048;           // row elements a rescan step reads
// Pre-final: when a piece of at least kPreFinalMin units is within kPreFinal
// stages of its end, the selectors sort what they hold, so that its end only
// merges the words of the last stages.
constexpr int kPreFinal = 8;
constexpr int kPreFinalMin = 16;
constexpr int kMaxSplit = 64;
constexpr uint32_t kWaitLimit = 1u << 22;    // polls before a wait gives up
// With TOPK_FLAG_TEST_STALL: every wait gives up after this many polls, and
// the producer stops for good in front of ring stage kTestStallStage (its
// barrier never completes), so that the waits behind it run out.
constexpr uint32_t kTestWaitLimit = 1u << 14;
constexpr int kTestStallStage = 3;

// Launch plan: one CTA per SM of the device, at most kMaxFlatCtas (results
// never depend on it).  A batch of at least as many rows as that count is not
// split.  Workspace sizes are computed for kMaxFlatCtas, the largest count a
// plan can use, so that they stay a function of the shape alone.
constexpr int kSmsDefault = 152;   // GB300's count: the plan when no device can be queried
constexpr int kMaxFlatCtas = 256;  // persistent grid cap (workspace slots)
constexpr int kMinFlatUnits = 16;  // a row is split into shares of at least 512 KB
constexpr int kMinSegUnits = 4;    // at least 128 KB per split segment

constexpr uint64_t kDefaultSeed = 0x5EEDC0DE1234ABCDull;

// ---------------------------------------------------------------------------
// Timeline (an instrumented build only: compiled with -DTOPK_TIMELINE=1 or 2).
// Each CTA of the selection kernel stamps the global timer at the events
// below into its row of g_timeline; with level 2 it also accumulates SM
// cycles per activity of one thread of each role (producer lane 0, filter
// warp 0 lane 0, selector thread 0).  topk_timeline_read copies the table
// out.  In the normal build every TL_* macro is empty and the table does not
// exist.
#ifndef TOPK_TIMELINE
#define TOPK_TIMELINE 0
#endif
constexpr int kTlSlots = 128;  // u64 slots per CTA
constexpr int kTlPieces = 4;    // pieces recorded per CTA
constexpr int kTlPerPiece = 16; // slots per piece
enum TlSlot : int {
  kTlStart = 0,       // kernel entry
  kTlSetup = 1,       // after the set-up barrier
  kTlFirstCopy = 2,   // producer: first copy issued
  kTlLastCopy = 3,    // producer: last copy issued
  kTlProdExit = 4,    // producer: done
  kTlFiltFirst = 5,   // filter warp 0: first stage taken (threshold in hand)
  kTlFiltExit = 6,    // filter warp 0: done
  kTlSelExit = 7,     // selectors: done
  kTlInfo = 8,        // SM id | pieces << 32
  kTlProdPiece = 9,   // producer: first piece planned
  kTlProdOrder = 10,  // producer: its first visiting order drawn
  kTlWarmEnter = 11,  // selectors: first warm start entered
  kTlWarmUnit0 = 12,  // ... its first unit read and the warps' keys shared
  kTlWarmCount = 13,  // ... the sample counted
  kTlWarmSecond = 14, // ... a second round counted (if one ran)
  kTlPiece0 = 16,     // per piece p: kTlPerPiece slots from kTlPiece0 + 16p:
                      //   +0 starting threshold published, +1 filter warp 0
                      //   takes its first stage, +2 filter group 0 (warp 0)
                      //   releases its last stage, +3 selectors done with it
                      //   (row written or partial list published; a leader
                      //   after its merge), +4 final tray sort and merge done,
                      //   +5 ticket taken, +6 leader: partner lists merged,
                      //   +7 pre-final sort done, +8 selectors see the piece's
                      //   filters done, +9 pre-final started, +10 final sort
                      //   done (before its merge), +11 partial list published
                      //   (before the ticket), +12 filter group 1 releases its
                      //   last stage, +13 producer: last copy issued
  kTlCyc0 = kTlPiece0 + kTlPieces * kTlPerPiece,  // cycle accumulators, see TlCyc
};
enum TlCyc : int {
  kCycFiltWaitFull = 0,  // filter warp 0: waiting for a stage to land
  kCycFiltWaitTheta,     // filter warp 0: waiting for a piece's starting threshold
  kCycFiltCand,          // filter warp 0: candidate path (classify, reserve, write)
  kCycFiltStages,        // filter warp 0: stages taken (a count)
  kCycFiltCandStages,    // filter warp 0: stages that took the candidate path (a count)
  kCycSelWarm,           // selectors: warm starts
  kCycSelTake,           // selectors: moving inbox words to the tray
  kCycSelPrune,          // selectors: prunes (select without sort)
  kCycSelSort,           // selectors: tray sorts and merges before a piece's end
  kCycSelEnd,            // selectors: piece ends (final sort, output or ticket, leader merge)
  kCycSelPoll,           // selectors: polling for work
  kCycSelLeader,         // selectors: leader merges (a count)
  kCycProdWaitEmpty,     // producer: waiting for a free ring stage
  kCycSelRescan,         // selectors: rescans (a count)
  kCycFiltBody,          // filter warp 0: a stage from landed to released
  kCycCandClassify,      // filter warp 0: candidate path, classifying the flagged groups
  kCycCandReserve,       // filter warp 0: candidate path, reserving inbox slots
  kCycCandWrite,         // filter warp 0: candidate path, writing the words
  kCycCandWords,         // filter warp 0: words its lanes wrote (a count)
  kCycFiltLoad,          // filter warp 0: a stage's loads and folded test (from landed)
  kCycCount
};
static_assert(kTlPiece0 + kTlPerPiece * kTlPieces <= kTlCyc0 && kTlCyc0 + kCycCount <= kTlSlots,
              "timeline slots");
// The short-row kernel's slots (its CTA's thread 0, SM cycles summed over the
// CTA's rows): rows, row start (queue item, row order and length, first
// loads issued), chunk loop without its selects, selects, row end (final
// select, sort, write), whole CTA, chunks, selects, waits for a chunk to land.
enum TlShort : int {
  kTlShortRows = 100, kTlShortMeta, kTlShortChunks, kTlShortSelect, kTlShortEnd, kTlShortTotal,
  kTlShortNChunks, kTlShortNSelects, kTlShortWait, kTlShortEndSlot
};
static_assert(kTlCyc0 + kCycCount <= kTlShortRows && kTlShortEndSlot <= kTlSlots, "timeline slots");

#if TOPK_TIMELINE
constexpr int kTlCtas = 512;   // CTAs recorded

__device__ __forceinline__ uint32_t smid() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ unsigned long long tl_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ unsigned long long g_timeline[kTlCtas * kTlSlots];
#define TL_SET(slot, v)                                                                  \
  do {                                                                                   \
    if (blockIdx.x < unsigned(kTlCtas)) g_timeline[blockIdx.x * kTlSlots + (slot)] = (v); \
  } while (0)
#define TL_PIECE(pc, off)                                   \
  do {                                                      \
    if ((pc) >= 0 && (pc) < kTlPieces) TL_SET(kTlPiece0 + kTlPerPiece * (pc) + (off), tl_now()); \
  } while (0)
#if TOPK_TIMELINE >= 2
// level 2: cycle accumulators as well (they slow the filter loop noticeably)
#define TL_CYCLES 1
#define TL_CYC_DECL(name) unsigned long long name[kCycCount] = {}
#define TL_CLK(var) const long long var = clock64()
#define TL_ACC(arr, which, since) ((arr)[which] += (unsigned long long)(clock64() - (since)))
#define TL_CNT(arr, which) (++(arr)[which])
#define TL_FLUSH(arr)                                                   \
  do {                                                                  \
    for (int q_ = 0; q_ < kCycCount; ++q_)                              \
      if ((arr)[q_]) TL_SET(kTlCyc0 + q_, (arr)[q_]);                   \
  } while (0)
#endif
#else
#define TL_SET(slot, v) ((void)0)
#define TL_PIECE(pc, off) ((void)0)
#endif
#ifndef TL_CYCLES
#define TL_CYCLES 0
#define TL_CYC_DECL(name) [[maybe_unused]] int name = 0
#define TL_CLK(var) ((void)0)
#define TL_ACC(arr, which, since) ((void)(arr))
#define TL_CNT(arr, which) ((void)(arr))
#define TL_FLUSH(arr) ((void)(arr))
#endif

// ---------------------------------------------------------------------------
// Bounds checks (the debug build only: compiled with -DTOPK_DEBUG_BOUNDS=1).
// IN_BOUNDS(cond, status) guards each shared- or global-memory write whose
// index is computed at run time (tray, kept list, leader-merge area, partial
// lists, outputs, block maxima, pool output): when cond is false the debug
// build sets TOPK_STATUS_BOUNDS and skips the write.  In the normal build it
// is the constant true.
#ifndef TOPK_DEBUG_BOUNDS
#define TOPK_DEBUG_BOUNDS 0
#endif
#if TOPK_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_ok(bool ok, uint32_t* status) {
  if (!ok) atomicOr(status, TOPK_STATUS_BOUNDS);
  return ok;
}
#define IN_BOUNDS(cond, status) bounds_ok((cond), (status))
#else
#define IN_BOUNDS(cond, status) true
#endif

// The CTA: filter warps, selector warps and one producer warp.
constexpr int kNF = 8;
constexpr int kNS = 8;
constexpr int kNFT = kNF * 32;                   // filter threads
constexpr int kFG = 2;                           // filter groups (alternate ring stages)
constexpr int kGW = kNF / kFG;                   // warps per filter group
constexpr int kGT = kGW * 32;                    // threads per filter group
constexpr int kNST = kNS * 32;                   // selector threads
constexpr int kThreads = kNFT + kNST + 32;
constexpr int kProducerWarp = kNF + kNS;
constexpr int kEPT = kUnit / kNFT;               // elements per filter thread per stage
constexpr int kF4 = kEPT / 4;                    // float4 loads per filter thread per stage
constexpr int kInbox = 2048;                     // words per inbox (two inboxes)
constexpr int kTray = 3072;                      // tray words
constexpr int kTable = 16;                       // piece descriptors in flight
// Inbox words the selectors move per step.  A take must never reach a slot
// reserved by a filter lane that is itself waiting for room, so it stays at
// least one lane-stage reservation (2 kEPT words: a filter lane tests 64
// elements of a stage) short of the inbox size.
constexpr int kTakeMax = (kInbox - 2 * kEPT) < 1024 ? (kInbox - 2 * kEPT) : 1024;
// Smallest batch the selectors take while the piece's filters are still
// running (a prune needs kPruneStep new words anyway); polling for less only
// takes issue slots from the filter warps.
constexpr int kTakeMin = 256;
static_assert(kEPT == 32, "one candidate bit per element of a thread's stage share");
static_assert((kInbox & (kInbox - 1)) == 0, "inbox ring size is a power of two");
static_assert(kTakeMax >= 256, "inbox leaves room for a take");
static_assert(kTray >= kTrayMark + 512 && kTray >= kTakeMax, "tray holds a take past its mark");
static_assert(kInbox + kTray >= 2 * TOPK_MAX_K, "leader merge holds two lists");

// Ring stages: five 32 KB stages when the kept list is small, four otherwise
// (shared memory is 227 KB per CTA).
__host__ __device__ inline int ring_stages(int kp) { return kp <= 512 ? 5 : 4; }

// Plans.
constexpr int kPlanItems = 0;  // (row, segment) items dealt round-robin to the grid
constexpr int kPlanFlat = 1;   // equal shares of the batch's units
constexpr int kPlanQueue = 2;  // (row, segment) items taken from a shared queue, longest rows first
constexpr int kQueueMaxUnits = 4096;  // longest row (in units) the queue's order kernel sorts

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)              header: u32 status
//   tickets   u32[rows]   split-row leader election, zero between calls
//   survivors u32[rows]   tray words that entered a bitonic tray sort, per row
//   sorts     u32[rows]   bitonic tray sorts per row
//   admitted  u32[rows]   elements that passed the threshold test, per row
//                         (the three counters accumulate until read)
//   queue     u32[2]      queue plan: next item, CTAs done; zero between calls
//   order     i32[rows]   queue plan: rows, longest first
//   theta     u64[rows]   split rows: best threshold word any of the row's CTAs
//                         has reached, zero between calls
//   spec      u64[rows]   split rows: largest speculative threshold word any of
//                         the row's pieces started from, zero between calls
//   partials  u64[slots][kp]  local top-k lists of split rows; slots =
//                         max(rows * split, 2 * kMaxFlatCtas) when rows can
//                         be split, else none
struct WsLayout {
  size_t tickets, survivors, sorts, admitted, queue, order, theta, spec, partials, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

bool shape_ok(int32_t rows, int64_t n, int32_t k) {
  return rows >= 0 && n >= 1 && n <= INT32_MAX && k >= 1 && k <= TOPK_MAX_K;
}

// CTAs per row of the automatic plan for `plan_sms` CTAs (the device's SM
// count, at most kMaxFlatCtas).
int32_t auto_split(int32_t rows, int64_t n, int plan_sms) {
  if (rows <= 0 || rows >= plan_sms) return 1;
  const int64_t m = (n + kUnit - 1) / kUnit;
  int64_t s = plan_sms / rows;
  const int64_t by_len = m / kMinSegUnits;
  if (s > by_len) s = by_len;
  if (s > kMaxSplit) s = kMaxSplit;
  if (s < 1) s = 1;
  return int32_t(s);
}

// Partial-list slots a call may need.  With the automatic plan a short batch
// may run either plan (the choice depends on whether lengths are passed).
size_t partial_slots(int32_t rows, int32_t split_arg, int32_t split, int plan_sms) {
  size_t slots = split > 1 ? size_t(rows) * size_t(split) : 0;
  if (split_arg == 0 && rows > 0 && rows < plan_sms) {
    const size_t flat = 2 * size_t(kMaxFlatCtas);
    if (flat > slots) slots = flat;
  }
  return slots;
}

WsLayout ws_layout(int32_t rows, int32_t kp, size_t slots) {
  WsLayout L;
  size_t off = 256;
  L.tickets = off;
  off = align256(off + sizeof(uint32_t) * size_t(rows));
  L.survivors = off;
  off = align256(off + sizeof(uint32_t) * size_t(rows));
  L.sorts = off;
  off = align256(off + sizeof(uint32_t) * size_t(rows));
  L.admitted = off;
  off = align256(off + sizeof(uint32_t) * size_t(rows));
  L.queue = off;
  off = align256(off + 2 * sizeof(uint32_t));
  L.order = off;
  off = align256(off + sizeof(int32_t) * size_t(rows));
  L.theta = off;
  off = align256(off + sizeof(uint64_t) * size_t(rows));
  L.spec = off;
  off = align256(off + sizeof(uint64_t) * size_t(rows));
  L.partials = off;
  off = align256(off + sizeof(uint64_t) * slots * size_t(kp));
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// Kernel parameters and shared-memory layout.

struct Params {
  const float* scores;
  int64_t row_stride;
  int64_t n;
  const int32_t* lengths;  // may be null
  int32_t rows;
  int32_t k;
  int32_t kp;         // next power of two >= k: kept-list capacity
  int32_t nstage;     // ring stages
  int32_t plan;       // kPlanItems, kPlanFlat or kPlanQueue
  int32_t split;      // items and queue plans: segments per row
  int32_t seg_units;  // items and queue plans: units per segment
  int32_t u_full;     // units per full row
  float* out_vals;
  int32_t* out_idx;
  uint32_t* status;
  uint32_t* tickets;
  uint32_t* survivors;
  uint32_t* sorts;
  uint32_t* admitted;
  unsigned long long* row_theta;
  unsigned long long* row_spec;
  uint64_t* partials;
  uint32_t seed_lo, seed_hi;
  uint32_t flags;
  uint32_t* queue;    // queue plan: next item, CTAs done
  const int32_t* order;  // queue plan: rows, longest first (null: index order)
  float* bmax;        // block pool: block maxima per row (null: not asked for)
  int64_t bstride;    // block pool: row stride of bmax, in blocks
  int64_t nslots;       // partial-list slots in the workspace
  uint32_t wait_limit;  // polls before a wait gives up
  int32_t stall_at;     // test only: ring stage the producer stops in front of (-1: none)
};

// What the producer tells the filters about a stage.
struct __align__(16) StageDesc {
  uint32_t e0;      // row-local index of the unit's first element
  uint32_t nvalid;  // valid elements in the unit (0 for an empty row)
  uint32_t r;       // row
  uint32_t tag;     // piece sequence number | kFirst | kLast | kLastG, or kEnd
};
constexpr uint32_t kSeqMask = 0x0FFFFFFFu;
constexpr uint32_t kFirst = 1u << 28;  // the piece's first stage
constexpr uint32_t kLast = 1u << 29;   // the piece's last stage
constexpr uint32_t kEnd = 1u << 30;    // no more stages
constexpr uint32_t kLastG = 1u << 31;  // a filter group's last stage of the piece (the
                                       // piece's last two stages, or its only one)

// A piece: units [u_begin, u_end) of row r, processed with one tray.
struct Piece {
  int32_t r;
  uint32_t L;            // valid length of the row
  int32_t u_begin, u_end;
  int32_t contributors;  // CTAs sharing the row (1 = unsplit)
  int32_t slot;          // partial slot when split
  int32_t first_cta;     // kPlanFlat: first CTA of the row
  int32_t self;          // this CTA's contributor index within the row
  uint32_t g_first;      // ring stage count at the piece's first stage
};

struct SmemLayout {
  int ring, desc, inbox0, tray, inbox1, kept, perm, hist, bars, total;
};

__host__ __device__ inline SmemLayout smem_layout(int kp) {
  const int ns = ring_stages(kp);
  SmemLayout L;
  int off = 0;
  L.ring = off;
  off += ns * kUnit * int(sizeof(float));
  L.desc = off;
  off += ns * int(sizeof(StageDesc));
  // inbox 0, tray and inbox 1 are contiguous: a leader merge uses its piece's
  // inbox plus the tray as one area
  L.inbox0 = off;
  off += kInbox * int(sizeof(uint64_t));
  L.tray = off;
  off += kTray * int(sizeof(uint64_t));
  L.inbox1 = off;
  off += kInbox * int(sizeof(uint64_t));
  L.kept = off;
  off += kp * int(sizeof(uint64_t));
  L.perm = off;
  off += kPermChunk * int(sizeof(uint32_t));
  L.hist = off;
  off += 256 * int(sizeof(uint32_t));
  L.bars = off;
  off += 2 * ns * int(sizeof(uint64_t));
  L.total = off;
  return L;
}

struct CtaState {
  uint32_t head[2];          // inbox p: next word the selectors take
  uint32_t tail[2];          // inbox p: next word a filter warp reserves
  int fdone[2];              // filter warps' stage reports for pieces of parity p (cumulative)
  int sel_pieces;            // pieces the selectors have finished
  int pieces_pub;            // piece descriptors the producer has published
  int npieces;               // total pieces of this CTA, -1 until known
  int flags;                 // selector broadcast scratch
  int cnt2;                  // compaction counter
  int leader;                // this CTA drew the last ticket
  int sel_b, sel_above, sel_binc;  // histogram select: chosen bin and counts
  int sel_n, sel_done;             // selector step: words to take, piece done
  uint32_t est[kNS];               // warm start: per selector warp key bound
  uint32_t est2[kNS];              // warm start: per selector warp candidate bound
  uint32_t warm_cnt;               // warm start: elements reaching the candidate
  uint32_t est3[kNS];              // warm start: per selector warp largest key
  uint32_t spec_cnt[5];            // warm start: sample counts of the speculative bounds
  uint32_t est4[kNS];              // warm start: per selector warp smallest unit maximum
  unsigned long long spec[2];      // speculative threshold word of the piece using inbox p
  const uint64_t* gsrc[16];        // leader merge: the partial lists of one gather step
  int warm_pub;                    // pieces whose starting threshold is set
  int warm_claim;                  // pieces whose starting threshold some role has taken on
  int first_issued;                // pieces whose first stage the producer has issued
  uint32_t fprog;                  // stages filter warp 0 has released
  int sel_pre;                     // selector step: pre-final due
  uint32_t wait_limit;             // polls before a wait gives up (the kernel's parameter)
  unsigned long long theta[2];     // threshold word of the piece using inbox p
  Piece table[kTable];             // piece descriptors, by sequence number
};

// Quotient of non-negative 64-bit values, with the (much shorter) 32-bit
// division when both fit: the plan arithmetic runs before a CTA's first copy.
__device__ __forceinline__ int64_t udiv(int64_t a, int64_t b) {
  if (((uint64_t(a) | uint64_t(b)) >> 32) == 0) return int64_t(uint32_t(a) / uint32_t(b));
  return a / b;
}
__device__ __forceinline__ int64_t flat_lo(int64_t g, int64_t M, int64_t G) { return udiv(g * M, G); }
__device__ __forceinline__ int32_t flat_cta_of(int64_t b, int64_t M, int64_t G) {
  return int32_t(udiv((b + 1) * G - 1, M));
}

// The next item of the queue plan's shared queue, taken by lane 0 for the
// warp; `total` or more means the queue is empty.  The last CTA to find it
// empty resets it for the next call (every other CTA has stopped taking
// items by then).  Kept out of line: it runs once per piece.
__device__ __noinline__ uint32_t queue_take(uint32_t* queue, uint32_t total) {
  uint32_t q = 0;
  if ((threadIdx.x & 31) == 0) {
    q = atomicAdd(queue, 1u);
    if (q >= total) {
      __threadfence();
      if (atomicAdd(queue + 1, 1u) == gridDim.x - 1u) {
        atomicExch(queue, 0u);
        atomicExch(queue + 1, 0u);
      }
    }
  }
  return __shfl_sync(0xFFFFFFFFu, q, 0);
}

// Piece w starts from its split row's shared words (rt proven, rs
// speculative; at least one is set): the role that claimed the piece
// publishes them as the piece's threshold.
__device__ __forceinline__ void adopt_row_theta(CtaState& st, int w, unsigned long long rt,
                                                unsigned long long rs) {
  if (rt != 0ull) atomicMax(&st.theta[w & 1], rt);
  if (rs > rt) {
    atomicMax(&st.theta[w & 1], rs);
    atomicMax(&st.spec[w & 1], rs);
  }
  __threadfence_block();
  atomicMax(&st.warm_pub, w + 1);
  TL_PIECE(w, 0);
}

// A filter warp's lane 0 at the first stage of piece seq: wait (at most
// `limit` polls) for the piece's starting threshold.  The selectors set it
// once its first units have landed, and only after piece seq - 2 (which used
// the same inbox, counters and threshold word) is finished.  A piece of a
// split row whose other CTAs already share a threshold need not wait for the
// selectors (they may still be finishing the piece before): once piece
// seq - 2 is finished, the filter warp that claims the piece first adopts
// the row's words itself.  Out of line: it runs once per piece.
__device__ __noinline__ bool filter_wait_theta(const unsigned long long* row_theta,
                                               const unsigned long long* row_spec, CtaState& st,
                                               int seq, uint32_t limit) {
  const Piece& pc = st.table[seq % kTable];
  for (uint32_t it = 0; *reinterpret_cast<volatile int*>(&st.warm_pub) < seq + 1; ++it) {
    if (it > limit) return false;
    if (pc.contributors > 1 && (it & 3u) == 0u &&
        *reinterpret_cast<volatile int*>(&st.sel_pieces) >= seq - 1 &&
        *reinterpret_cast<volatile int*>(&st.warm_claim) == seq) {
      const unsigned long long rt = *reinterpret_cast<const volatile unsigned long long*>(&row_theta[pc.r]);
      const unsigned long long rs = *reinterpret_cast<const volatile unsigned long long*>(&row_spec[pc.r]);
      if ((rt | rs) != 0ull && atomicCAS(&st.warm_claim, seq, seq + 1) == seq) {
        adopt_row_theta(st, seq, rt, rs);
        return true;
      }
    }
    __nanosleep(200);
  }
  return true;
}

// The pi-th piece of this CTA: 0 = no more pieces, 1 = a piece, 2 = an
// empty item to skip (a segment past the end of a short row).
__device__ int get_piece(const Params& p, int32_t pi, Piece& out, bool& bad_len) {
  const int64_t cta = blockIdx.x;
  const int64_t G = gridDim.x;
  bad_len = false;
  if (p.plan == kPlanItems || p.plan == kPlanQueue) {
    const int64_t total = int64_t(p.rows) * p.split;
    int64_t item;
    if (p.plan == kPlanItems) {
      item = cta + int64_t(pi) * G;  // dealt round-robin
    } else {
      item = int64_t(queue_take(p.queue, uint32_t(total)));
    }
    if (item >= total) return 0;
    const int32_t rank = int32_t(udiv(item, p.split));
    const int32_t r = p.order ? p.order[rank] : rank;
    const int32_t s = int32_t(item - int64_t(rank) * p.split);
    int64_t L = p.lengths ? int64_t(p.lengths[r]) : p.n;
    if (L < 0 || L > p.n) {
      bad_len = s == 0;  // a1: reported once per row
      L = L < 0 ? 0 : p.n;
    }
    const int32_t m = int32_t((L + kUnit - 1) / kUnit);
    const int32_t contributors = m == 0 ? 1 : (m + p.seg_units - 1) / p.seg_units;
    if (s >= contributors) return 2;
    out.r = r;
    out.L = uint32_t(L);
    out.u_begin = s * p.seg_units;
    out.u_end = m == 0 ? 0 : min(m, out.u_begin + p.seg_units);
    out.contributors = contributors;
    out.slot = r * p.split + s;
    out.first_cta = 0;
    out.self = s;
    return 1;
  }
  const int64_t M = int64_t(p.rows) * p.u_full;
  const int64_t lo = flat_lo(cta, M, G), hi = flat_lo(cta + 1, M, G);
  const int64_t r0 = udiv(lo, p.u_full);
  const int64_t r = r0 + pi;
  const int64_t rs = r * p.u_full;
  if (r >= p.rows || rs >= hi) return 0;
  out.r = int32_t(r);
  out.L = uint32_t(p.n);
  out.u_begin = int32_t(lo > rs ? lo - rs : 0);
  out.u_end = int32_t(hi - rs < p.u_full ? hi - rs : p.u_full);
  const int32_t g0 = flat_cta_of(rs, M, G), g1 = flat_cta_of(rs + p.u_full - 1, M, G);
  out.contributors = g1 - g0 + 1;
  out.first_cta = g0;
  out.self = int32_t(cta) - g0;
  out.slot = 2 * int32_t(cta) + (r == r0 ? 0 : 1);
  return 1;
}

// Visiting order of `m` <= kPermChunk consecutive units of row `row`
// starting at unit `first`, drawn by one warp: the units sorted by a Philox
// draw whose low 8 bits are replaced by the unit's position, so the order is
// a permutation whatever the draws and never depends on the scores.
// perm[i] & 255 = position visited i-th.  The sort runs over 32E keys (E
// the smallest power of two with 32E >= m, empty keys last); key i sits in
// lane i % 32, register i / 32; strides of 32 and more swap registers,
// shorter ones exchange through shuffles.
template <int E>
__device__ __forceinline__ void visit_keys(uint32_t (&v)[E], int m, int64_t first, int32_t row,
                                           uint32_t seed_lo, uint32_t seed_hi, bool identity,
                                           int lane) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = e * 32 + lane;
    uint32_t key = 0xFFFFFFFFu;
    if (j < m) {
      if (identity) {
        key = uint32_t(j);
      } else {
        const uint4 r = philox4x32_10(make_uint4(uint32_t(first + j), uint32_t(row), 0u, 0u),
                                      seed_lo, seed_hi);
        key = (r.x & ~uint32_t(kPermChunk - 1)) | uint32_t(j);
      }
    }
    v[e] = key;
  }
}

template <int E>
__device__ __forceinline__ void visit_order_sort(uint32_t* perm, int m, int64_t first, int32_t row,
                                                 uint32_t seed_lo, uint32_t seed_hi,
                                                 bool identity, int lane) {
  constexpr int n = 32 * E;
  uint32_t v[E];
  visit_keys<E>(v, m, first, row, seed_lo, seed_hi, identity, lane);
#pragma unroll
  for (int size = 2; size <= n; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32) {
        const int es = stride >> 5;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & es) == 0) {
            const bool up = ((e * 32 + lane) & size) == 0;
            const uint32_t a = v[e], b = v[e | es];
            const bool sw = (a > b) == up;
            v[e] = sw ? b : a;
            v[e | es] = sw ? a : b;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, v[e], stride);
          const bool up = ((e * 32 + lane) & size) == 0;
          const bool lower = (lane & stride) == 0;
          v[e] = (lower == up) ? min(v[e], o) : max(v[e], o);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) perm[e * 32 + lane] = v[e];
  __syncwarp();
}

__device__ void build_visit_order_warp(uint32_t* perm, int m, int64_t first, int32_t row,
                                       uint32_t seed_lo, uint32_t seed_hi, bool identity,
                                       int lane) {
  static_assert(kPermChunk == 256, "orders of up to 8 keys per lane");
  if (m <= 32) visit_order_sort<1>(perm, m, first, row, seed_lo, seed_hi, identity, lane);
  else if (m <= 64) visit_order_sort<2>(perm, m, first, row, seed_lo, seed_hi, identity, lane);
  else if (m <= 128) visit_order_sort<4>(perm, m, first, row, seed_lo, seed_hi, identity, lane);
  else visit_order_sort<8>(perm, m, first, row, seed_lo, seed_hi, identity, lane);
}

// The first nhead entries of the same order (its nhead smallest keys), found
// by warp minima without the sort, into perm[0, nhead): nhead <= m <= 64.
// The keys are distinct (their low bits are the positions), so the q-th
// smallest is the smallest key above the (q-1)-th.
__device__ void visit_order_head(uint32_t* perm, int m, int64_t first, int32_t row,
                                 uint32_t seed_lo, uint32_t seed_hi, bool identity, int lane,
                                 int nhead) {
  uint32_t v[2];
  visit_keys<2>(v, m, first, row, seed_lo, seed_hi, identity, lane);
  uint32_t prev = 0u;
  for (int q = 0; q < nhead; ++q) {
    uint32_t lm = 0xFFFFFFFFu;
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (q == 0 || v[e] > prev) lm = min(lm, v[e]);
    prev = __reduce_min_sync(0xFFFFFFFFu, lm);
    if (lane == 0) perm[q] = prev;
  }
  __syncwarp();
}

// Bitonic network, largest first, over the n = T::size * E words a[0, n),
// held in registers while it runs: thread t keeps words tE .. tE+E-1.
// Strides below E compare registers of one thread, strides below 32E
// exchange through warp shuffles, longer strides (between warps) go through
// the array with two team barriers each.  Merge levels below first_size are
// skipped: first_size = 2 sorts, first_size = n merges one bitonic
// sequence.  The caller has made a[] visible to the team; the result is
// stored back and followed by a team barrier.
template <class T, int E>
__device__ void team_bitonic(uint64_t* a, int first_size, int t) {
  constexpr int n = T::size * E;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = a[t * E + e];
#pragma unroll
  for (int size = 2; size <= n; size <<= 1) {
    if (size < first_size) continue;
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & stride) == 0) {
            const bool larger_first = ((t * E + e) & size) == 0;
            const uint64_t x = v[e], y = v[e | stride];
            const bool sw = larger_first ? (x < y) : (x > y);
            v[e] = sw ? y : x;
            v[e | stride] = sw ? x : y;
          }
        }
      } else if (stride < 32 * E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = t * E + e;
          const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v[e], stride / E);
          const bool keep_max = ((i & stride) == 0) == ((i & size) == 0);
          v[e] = keep_max ? (v[e] > o ? v[e] : o) : (v[e] < o ? v[e] : o);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) a[t * E + e] = v[e];
        T::sync();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = t * E + e;
          const uint64_t o = a[i ^ stride];
          const bool keep_max = ((i & stride) == 0) == ((i & size) == 0);
          v[e] = keep_max ? (v[e] > o ? v[e] : o) : (v[e] < o ? v[e] : o);
        }
        T::sync();
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) a[t * E + e] = v[e];
  T::sync();
}

// Largest-first bitonic network over n (a power of two) words of a[]:
// first_size = 2 sorts, first_size = n merges a bitonic sequence.  Ends with
// a team barrier.
template <class T>
__device__ void team_sort_desc(uint64_t* a, int n, int first_size, int t) {
  static_assert(T::size == 256, "register networks are laid out for 256 threads");
  if (n == 256) team_bitonic<T, 1>(a, first_size, t);
  else if (n == 512) team_bitonic<T, 2>(a, first_size, t);
  else if (n == 1024) team_bitonic<T, 4>(a, first_size, t);
  else bitonic_network<T, uint64_t, true>(a, n, first_size, 1, 0, t);
}

// Merge a sorted-descending `batch` of n words (read as if padded with empty
// words to kp) into the kept list: the best kp of both end up sorted in kept.
template <class T>
__device__ void merge_into_kept(uint64_t* kept, const uint64_t* batch, int n, int kp, int t) {
  for (int j = t; j < kp; j += T::size) {
    const int i = kp - 1 - j;
    const uint64_t a = kept[j], b = i < n ? batch[i] : 0ull;
    kept[j] = a > b ? a : b;
  }
  T::sync();
  team_sort_desc<T>(kept, kp, kp, t);
}

__device__ __forceinline__ void write_row(const Params& p, int32_t r, const uint64_t* kept, int t,
                                          int nt) {
  float* ov = p.out_vals + int64_t(r) * p.k;
  int32_t* oi = p.out_idx + int64_t(r) * p.k;
  for (int j = t; j < p.k; j += nt) {
    const uint64_t w = kept[j];
    if (!IN_BOUNDS(r >= 0 && r < p.rows, p.status)) break;
    if (w == 0ull) {
      ov[j] = -__int_as_float(0x7F800000);
      oi[j] = -1;
    } else {
      ov[j] = key_to_float(uint32_t(w >> 32));
      oi[j] = int32_t(~uint32_t(w));
    }
  }
}

// One thread's share of a span of T * 32 elements read by T threads:
// elements 4 * (t + T u) + c, u < 8, c < 4.  A full, aligned span is read
// from shared memory only; otherwise elements past the copied prefix come
// from global memory and elements past the span's end are marked invalid
// (bit e of the result clear).  (T = 256: the selector team's view of a
// whole unit; T = 128: a filter group's view of half a unit.)
template <int T = kNFT>
__device__ __forceinline__ uint32_t load_share(float (&x)[kEPT], const float* src, const float* row,
                                               uint32_t e0, uint32_t nvalid, uint32_t copied,
                                               int t) {
  if (copied == uint32_t(T * kEPT)) {
#pragma unroll
    for (int u = 0; u < kF4; ++u) {
      const float4 v = reinterpret_cast<const float4*>(src)[t + T * u];
      x[4 * u + 0] = v.x;
      x[4 * u + 1] = v.y;
      x[4 * u + 2] = v.z;
      x[4 * u + 3] = v.w;
    }
    return 0xFFFFFFFFu;
  }
  uint32_t valid = 0u;
#pragma unroll
  for (int u = 0; u < kF4; ++u) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t pos = uint32_t(4 * (t + T * u) + c);
      float v = 0.f;
      if (pos < copied) v = src[pos];
      else if (pos < nvalid) v = __ldg(row + e0 + pos);
      x[4 * u + c] = v;
      valid |= uint32_t(pos < nvalid) << (4 * u + c);
    }
  }
  return valid;
}

// Warm start.  A key T (its low 16 bits zero) that at least m valid,
// non-NaN elements reach is a valid starting threshold word (T << 32) - 1
// for a piece once m * 8 = k of the piece's elements are known to reach the
// smallest of the eight warps' keys.  Each warp searches a 4-ary way over key
// bits 31..16: a step tries three keys and counts, warp-wide, the elements
// at or above each (the three counts packed into one reduction).

// Key of element e of a thread's share, or 0 for padding and NaN.
__device__ __forceinline__ uint32_t share_key(const float (&x)[kEPT], uint32_t valid, int e) {
  const uint32_t bits = __float_as_uint(x[e]);
  const bool use = ((valid >> e) & 1u) && (bits & 0x7FFFFFFFu) <= 0x7F800000u;
  return use ? order_key(bits) : 0u;
}

// For m <= 64 the counts run over the union of every lane's four largest
// keys of one unit (128 values per warp): T is reached by at least m real
// elements, and falls short of the exact bound only when some lane holds
// more than four of the warp's top m.  Lane lists are kept sorted,
// l0 >= l1 >= l2 >= l3; padding and NaN have key 0 and never count.
struct Top4 {
  uint32_t l0 = 0, l1 = 0, l2 = 0, l3 = 0;
  static __device__ __forceinline__ uint32_t key_of(float x) {
    const uint32_t bits = __float_as_uint(x);
    return (bits & 0x7FFFFFFFu) <= 0x7F800000u ? order_key(bits) : 0u;
  }
  __device__ __forceinline__ void add(uint32_t v) {
    const uint32_t a3 = max(l3, min(l2, v));
    const uint32_t a2 = max(l2, min(l1, v));
    const uint32_t a1 = max(l1, min(l0, v));
    l0 = max(l0, v);
    l1 = a1;
    l2 = a2;
    l3 = a3;
  }
  // four elements: sort them (five compare-exchanges), then the top four of
  // both sorted lists are max(l_i, g_{3-i}), a bitonic sequence that two
  // rounds of compare-exchanges sort
  __device__ __forceinline__ void add4(float4 f) {
    uint32_t a = key_of(f.x), b = key_of(f.y), c = key_of(f.z), d = key_of(f.w);
    auto cx = [](uint32_t& x, uint32_t& y) {
      const uint32_t hi = max(x, y), lo = min(x, y);
      x = hi;
      y = lo;
    };
    cx(a, b);
    cx(c, d);
    cx(a, c);
    cx(b, d);
    cx(b, c);
    uint32_t m0 = max(l0, d), m1 = max(l1, c), m2 = max(l2, b), m3 = max(l3, a);
    cx(m0, m2);
    cx(m1, m3);
    cx(m0, m1);
    cx(m2, m3);
    l0 = m0;
    l1 = m1;
    l2 = m2;
    l3 = m3;
  }
  __device__ __forceinline__ uint32_t count_ge(uint32_t t) const {
    return (l0 >= t ? 1u : 0u) + (l1 >= t ? 1u : 0u) + (l2 >= t ? 1u : 0u) + (l3 >= t ? 1u : 0u);
  }
  // Two searches at once (targets m1, m2), six trial keys per step, their
  // counts packed into two reductions.
  __device__ __forceinline__ void bound2(int m1, int m2, uint32_t& T1, uint32_t& T2) const {
    const uint32_t mm1 = uint32_t(m1), mm2 = uint32_t(m2);
    T1 = 0;
    T2 = 0;
#pragma unroll 1
    for (int b = 31; b >= 17; b -= 2) {
      uint32_t pk1 = 0, pk2 = 0;  // three counts of at most 128 each, eight bits each
#pragma unroll
      for (uint32_t i = 1; i <= 3; ++i) {
        pk1 += count_ge(T1 | (i << (b - 1))) << (8 * (i - 1));
        pk2 += count_ge(T2 | (i << (b - 1))) << (8 * (i - 1));
      }
      pk1 = __reduce_add_sync(0xFFFFFFFFu, pk1);
      pk2 = __reduce_add_sync(0xFFFFFFFFu, pk2);
      const uint32_t i1 = ((pk1 >> 16) & 0xFFu) >= mm1 ? 3u
                          : ((pk1 >> 8) & 0xFFu) >= mm1 ? 2u
                          : (pk1 & 0xFFu) >= mm1 ? 1u : 0u;
      const uint32_t i2 = ((pk2 >> 16) & 0xFFu) >= mm2 ? 3u
                          : ((pk2 >> 8) & 0xFFu) >= mm2 ? 2u
                          : (pk2 & 0xFFu) >= mm2 ? 1u : 0u;
      T1 |= i1 << (b - 1);
      T2 |= i2 << (b - 1);
    }
  }
};

// The warp's exact R-th largest key over its elements (as warp_key_bound
// with low = 1: the largest T that at least R keys reach; 0 if fewer than R
// are valid), for a small R: the warp takes its largest key value below the
// last one taken, R times at most, counting the elements equal to it, until
// R elements have been taken -- R rounds of one pass instead of sixteen
// bisection rounds.
__device__ __forceinline__ uint32_t warp_rank_key(const float (&x)[kEPT], uint32_t valid, int R) {
  uint32_t key[kEPT];
#pragma unroll
  for (int e = 0; e < kEPT; ++e) key[e] = share_key(x, valid, e);
  uint32_t taken = 0, prev = 0xFFFFFFFFu;  // (no key is all ones: +inf's is 0xFF800000)
  for (int it = 0; it < R; ++it) {
    uint32_t lm = 0u;
#pragma unroll
    for (int e = 0; e < kEPT; ++e) lm = max(lm, key[e] < prev ? key[e] : 0u);
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, lm);
    if (m == 0u) return 0u;  // fewer than R valid elements
    uint32_t c = 0u;
#pragma unroll
    for (int e = 0; e < kEPT; ++e) c += key[e] == m ? 1u : 0u;
    taken += __reduce_add_sync(0xFFFFFFFFu, c);
    if (taken >= uint32_t(R)) return m;
    prev = m;
  }
  return 0u;  // (not reached: every round takes at least one element)
}

// For m > 64 the counts run over all 32 keys of each lane (one unit).  The
// bound resolves the key down to bit `low` (17: a 16-bit prefix; 1: the exact
// m-th key).
__device__ __forceinline__ uint32_t warp_key_bound(const float (&x)[kEPT], uint32_t valid, int m,
                                                   int low = 17) {
  uint32_t key[kEPT];
  uint32_t ok = 0;
#pragma unroll
  for (int e = 0; e < kEPT; ++e) {
    key[e] = share_key(x, valid, e);
    ok += key[e] != 0u ? 1u : 0u;
  }
  if (__reduce_add_sync(0xFFFFFFFFu, ok) < uint32_t(m)) return 0u;
  const uint32_t mm = uint32_t(m);
  uint32_t T = 0;
#pragma unroll 1
  for (int b = 31; b >= low; b -= 2) {
    const uint32_t t1 = T | (1u << (b - 1)), t2 = T | (2u << (b - 1)), t3 = T | (3u << (b - 1));
    uint32_t c12 = 0, c3 = 0;  // counts of at most 1024: two per word, sixteen bits each
#pragma unroll
    for (int e = 0; e < kEPT; ++e) {
      c12 += (key[e] >= t1 ? 1u : 0u) + (key[e] >= t2 ? 0x10000u : 0u);
      c3 += key[e] >= t3 ? 1u : 0u;
    }
    c12 = __reduce_add_sync(0xFFFFFFFFu, c12);
    c3 = __reduce_add_sync(0xFFFFFFFFu, c3);
    const uint32_t i = c3 >= mm ? 3u : (c12 >> 16) >= mm ? 2u : (c12 & 0xFFFFu) >= mm ? 1u : 0u;
    T |= i << (b - 1);
  }
  return T;
}

// The sample count a speculative start needs (2.5 k * sample / row length).
__host__ __device__ inline uint64_t spec_need(int k, int wu, uint32_t L) {
  const uint64_t sample = uint64_t(wu) * uint64_t(kUnit);
  return (5ull * uint64_t(k) * sample + 2ull * L - 1ull) / (2ull * L);
}

// The full warm-start sample of a piece, in units: kWarmUnitsSmallK when each
// selector warp needs at most 64 elements (k <= 512), else kWarmUnits.
__host__ __device__ inline int warm_cap(int k) {
  return (k + kNS - 1) / kNS <= 64 ? kWarmUnitsSmallK : kWarmUnits;
}

// Units a piece's warm start reads: warm_cap (at most the piece's units) for
// k <= 512; above that, kWarmUnits only where a speculative start may be
// taken (a long row), else one.
__host__ __device__ inline int warm_units(int k, int nu, uint32_t L) {
  const int cap = warm_cap(k);
  const int w = nu < 1 ? 1 : (nu < cap ? nu : cap);
  if ((k + kNS - 1) / kNS <= 64) return w;
  return (w == kWarmUnits && L > 0u && spec_need(k, w, L) <= kSpecMaxNeed) ? w : 1;
}

// Warm start of piece w, whose first units have landed in the ring (the
// filters hold them until the threshold is set), run by the selector team:
// each selector warp bounds its share of those units, the smallest bound is
// reached by at least k elements of the piece.  The piece may use the
// threshold word of its parity: the piece before it in that parity is
// finished.  A function of its own (not inlined), so that the lane lists
// keep registers instead of competing with the selector loop's state.
// Returns false if a wait gave up.
__device__ __noinline__ bool warm_start_piece(const float* scores, int64_t row_stride,
                                              unsigned long long* row_theta,
                                              unsigned long long* row_spec, CtaState& st,
                                              int w, const float* ring, const StageDesc* desc,
                                              uint64_t* full, int nstage, int k, int stt) {
#define wl (*reinterpret_cast<volatile uint32_t*>(&st.wait_limit))
  using Sel = Team<kNST, 1>;
  const int lane = stt & 31, swarp = stt >> 5;
  const int m_warm = (k + kNS - 1) / kNS;
  bool ok = true;
  const Piece pw = st.table[w % kTable];
  const int wu = warm_units(k, pw.u_end - pw.u_begin, pw.L);
  const float* wrow = scores + int64_t(pw.r) * row_stride;
  const bool waligned = (reinterpret_cast<uintptr_t>(wrow) & 15u) == 0;
  auto stage_of = [&](int q, const float*& src, StageDesc& d, uint32_t& copied) {
    const uint32_t g = pw.g_first + uint32_t(q);
    const int slot = int(g % uint32_t(nstage));
    // every reader observes the copy's completion itself (already complete)
    if (!mbar_wait(&full[slot], (g / uint32_t(nstage)) & 1u, wl)) ok = false;
    d = desc[slot];
    src = ring + slot * kUnit;
    copied = waligned ? (d.nvalid & ~3u) : 0u;
  };
  if (stt == 0) st.warm_cnt = 0u;
  if (stt == 0 && w == 0) TL_SET(kTlWarmEnter, tl_now());
  uint32_t mk = 0u;
  uint64_t spec = 0ull;  // speculative threshold word (0: none)
  bool decided = false;
  uint32_t mk_floor = 0u;  // a proven bound from the speculative candidates
  // Speculative start (pieces of long rows): the 8th, 7th and 6th largest of
  // the selector warps' rank-R keys in the first unit are candidates (R = 1,
  // the largest, for k <= 512; above, R makes the candidates' expected sample
  // count about 1.25 need);
  // the highest one that the wu sample units hold at least `need` elements
  // at or above is taken (need = 2.5 k * sample / row length, so that the row
  // holds about 3.6 k above it).  The count is a strict float compare (it
  // never counts NaN, and misses only -0.0 against a +0.0 bound).  Only when
  // no candidate is supported do the lane lists below run.
  const int nu = pw.u_end - pw.u_begin;
  if (wu == warm_cap(k) && nu >= wu) {
    const uint64_t need64 = spec_need(k, wu, pw.L);
    // (with the three-unit sample only the warps' largest keys are tried:
    // rank-R candidates need an exact per-warp select that costs more than a
    // speculative start saves on rows this short)
    if (need64 <= (wu == kWarmUnits ? uint64_t(kSpecMaxNeed) : 128ull)) {
      const uint32_t need = uint32_t(need64);
      const int R = need <= 128u ? 1 : int((5u * need + 4u * wu * kNS - 1u) / (4u * wu * kNS));
      float lm = -__int_as_float(0x7F800000);
      uint32_t wkey = 0u;  // this warp's rank-R key of the first unit
      {
        const float* src;
        StageDesc d;
        uint32_t copied;
        stage_of(0, src, d, copied);
        if (R > 1) {
          float x[kEPT];
          const uint32_t valid = load_share(x, src, wrow, d.e0, d.nvalid, copied, stt);
          wkey = warp_rank_key(x, valid, R);  // exact: a coarse bound could pass a whole top unit
        } else if (copied == uint32_t(kUnit)) {
#pragma unroll
          for (int u = 0; u < kF4; ++u) {
            const float4 v = reinterpret_cast<const float4*>(src)[stt + kNST * u];
            lm = fmaxf(lm, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
          }
        } else {
          for (int u = 0; u < kF4; ++u) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t pos = uint32_t(4 * (stt + kNST * u) + c);
              if (pos < copied) lm = fmaxf(lm, src[pos]);
              else if (pos < d.nvalid) lm = fmaxf(lm, __ldg(wrow + d.e0 + pos));
            }
          }
        }
      }
      if (R == 1) wkey = __reduce_max_sync(0xFFFFFFFFu, Top4::key_of(lm));
      if (lane == 0) st.est3[swarp] = wkey;
      if (stt == 0) {
        st.spec_cnt[0] = 0u;
        st.spec_cnt[1] = 0u;
        st.spec_cnt[2] = 0u;
        st.spec_cnt[3] = 0u;
        st.spec_cnt[4] = 0u;
      }
      Sel::sync();
      if (stt == 0 && w == 0) TL_SET(kTlWarmUnit0, tl_now());
      // the three smallest warp maxima
      uint32_t s8 = 0xFFFFFFFFu, s7 = 0xFFFFFFFFu, s6 = 0xFFFFFFFFu;
#pragma unroll
      for (int q = 0; q < kNS; ++q) {
        const uint32_t v = st.est3[q];
        const uint32_t n8 = min(s8, v), n7 = min(s7, max(s8, v)), n6 = min(s6, max(s7, v));
        s8 = n8;
        s7 = n7;
        s6 = n6;
      }
      if (s8 > 1u) {  // (every warp saw a value)
        const float f8 = key_to_float(s8 - 1u), f7 = key_to_float(s7 - 1u),
                    f6 = key_to_float(s6 - 1u);  // key >= s  <=>  value > key_to_float(s - 1)
        uint32_t ca = 0u, cb = 0u;               // counts: s8 | s7 << 16, and s6
        uint32_t umin = 0xFFFFFFFFu;             // smallest of this warp's unit maxima
        uint32_t ca0 = 0u, cb0 = 0u;             // the first unit's share of the counts
        for (int q = 0; q < wu; ++q) {
          const float* src;
          StageDesc d;
          uint32_t copied;
          stage_of(q, src, d, copied);
          float um = -__int_as_float(0x7F800000);
          if (copied == uint32_t(kUnit)) {
#pragma unroll 4
            for (int u = 0; u < kF4; ++u) {
              const float4 v = reinterpret_cast<const float4*>(src)[stt + kNST * u];
              const float vv[4] = {v.x, v.y, v.z, v.w};
              um = fmaxf(um, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                ca += (vv[c] > f8 ? 1u : 0u) + (vv[c] > f7 ? 0x10000u : 0u);
                cb += vv[c] > f6 ? 1u : 0u;
              }
            }
          } else {
            for (int u = 0; u < kF4; ++u) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint32_t pos = uint32_t(4 * (stt + kNST * u) + c);
                float v = -__int_as_float(0x7F800000);
                if (pos < copied) v = src[pos];
                else if (pos < d.nvalid) v = __ldg(wrow + d.e0 + pos);
                um = fmaxf(um, v);
                ca += (v > f8 ? 1u : 0u) + (v > f7 ? 0x10000u : 0u);
                cb += v > f6 ? 1u : 0u;
              }
            }
          }
          umin = min(umin, __reduce_max_sync(0xFFFFFFFFu, Top4::key_of(um)));
          if (q == 0) {
            ca0 = ca;
            cb0 = cb;
          }
        }
        ca = __reduce_add_sync(0xFFFFFFFFu, ca);
        cb = __reduce_add_sync(0xFFFFFFFFu, cb);
        ca0 = __reduce_add_sync(0xFFFFFFFFu, ca0);
        cb0 = __reduce_add_sync(0xFFFFFFFFu, cb0);
        if (lane == 0) {
          atomicAdd(&st.spec_cnt[0], ca);
          atomicAdd(&st.spec_cnt[1], cb);
          atomicAdd(&st.spec_cnt[3], ca0);
          atomicAdd(&st.spec_cnt[4], cb0);
          st.est4[swarp] = umin;
        }
        Sel::sync();
        if (stt == 0 && w == 0) TL_SET(kTlWarmCount, tl_now());
        const uint32_t n8 = st.spec_cnt[0] & 0xFFFFu, n7 = st.spec_cnt[0] >> 16,
                       n6 = st.spec_cnt[1];
        // the other sample units (not the first, where the candidates come
        // from) must hold at least half of it: a first unit that holds the
        // row's top (a sorted row) supports no speculation by itself
        const uint32_t o8 = n8 - (st.spec_cnt[3] & 0xFFFFu), o7 = n7 - (st.spec_cnt[3] >> 16),
                       o6 = n6 - st.spec_cnt[4];
        const uint32_t half = (need + 1u) / 2u;
        uint32_t sk = 0u, nk = 0u;
        if (n6 >= need && (o6 >= half || n6 >= uint32_t(k))) {
          sk = s6;
          nk = n6;
        } else if (n7 >= need && (o7 >= half || n7 >= uint32_t(k))) {
          sk = s7;
          nk = n7;
        } else if (n8 >= need && (o8 >= half || n8 >= uint32_t(k))) {
          sk = s8;
          nk = n8;
        }
        if (sk == 0u && R == 1) {
          // Second round: the smallest of the 8 wu (warp, unit) maxima of the
          // sample, a lower candidate, counted the same way.
          uint32_t s2 = 0xFFFFFFFFu;
#pragma unroll
          for (int q = 0; q < kNS; ++q) s2 = min(s2, st.est4[q]);
          if (s2 > 1u && s2 < s8) {
            const float f2 = key_to_float(s2 - 1u);
            uint32_t c2 = 0u;
            for (int q = 0; q < wu; ++q) {
              const float* src;
              StageDesc d;
              uint32_t copied;
              stage_of(q, src, d, copied);
              if (copied == uint32_t(kUnit)) {
#pragma unroll 4
                for (int u = 0; u < kF4; ++u) {
                  const float4 v = reinterpret_cast<const float4*>(src)[stt + kNST * u];
                  c2 += (v.x > f2 ? 1u : 0u) + (v.y > f2 ? 1u : 0u) + (v.z > f2 ? 1u : 0u) +
                        (v.w > f2 ? 1u : 0u);
                }
              } else {
                for (int u = 0; u < kF4; ++u) {
#pragma unroll
                  for (int c = 0; c < 4; ++c) {
                    const uint32_t pos = uint32_t(4 * (stt + kNST * u) + c);
                    float v = -__int_as_float(0x7F800000);
                    if (pos < copied) v = src[pos];
                    else if (pos < d.nvalid) v = __ldg(wrow + d.e0 + pos);
                    c2 += v > f2 ? 1u : 0u;
                  }
                }
              }
            }
            c2 = __reduce_add_sync(0xFFFFFFFFu, c2);
            if (lane == 0) atomicAdd(&st.spec_cnt[2], c2);
            Sel::sync();
            if (stt == 0 && w == 0) TL_SET(kTlWarmSecond, tl_now());
            if (st.spec_cnt[2] >= need) {
              sk = s2;
              nk = st.spec_cnt[2];
            }
          }
        }
        if (sk != 0u) {
          // A candidate the sample alone shows k elements above is proven:
          // a floor for the bounds below (which may find a higher one).
          if (nk >= uint32_t(k)) {
            mk_floor = sk;
          } else {
            spec = (uint64_t(sk) << 32) - 1ull;
            decided = true;
          }
        }
      }
    }
  }
  if (!decided) {
    if (m_warm > 64) {
      // one unit, all 32 keys of every lane
      const float* src;
      StageDesc d;
      uint32_t copied;
      stage_of(0, src, d, copied);
      float x[kEPT];
      const uint32_t valid = load_share(x, src, wrow, d.e0, d.nvalid, copied, stt);
      const uint32_t est = warp_key_bound(x, valid, m_warm);
      if (lane == 0) st.est[swarp] = est;
      Sel::sync();
      mk = 0xFFFFFFFFu;
#pragma unroll
      for (int q = 0; q < kNS; ++q) mk = min(mk, st.est[q]);
    } else {
      // Lane lists of the first unit give two bounds per warp: a safe one
      // (m elements of the unit) and a candidate for all wu units (about
      // 1.25 m / wu elements of the unit).  The candidate is taken if a count
      // finds k elements at or above it: the lane lists' count in the first
      // unit (a lower bound) plus a strict float compare over the other units
      // (it never counts NaN, and misses only -0.0 against a +0.0 bound).
      Top4 top;
      {
        const float* src;
        StageDesc d;
        uint32_t copied;
        stage_of(0, src, d, copied);
        if (copied == uint32_t(kUnit)) {
#pragma unroll 2
          for (int u = 0; u < kF4; ++u) top.add4(reinterpret_cast<const float4*>(src)[stt + kNST * u]);
        } else {
          for (int u = 0; u < kF4; ++u) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t pos = uint32_t(4 * (stt + kNST * u) + c);
              if (pos < copied) top.add(Top4::key_of(src[pos]));
              else if (pos < d.nvalid) top.add(Top4::key_of(__ldg(wrow + d.e0 + pos)));
            }
          }
        }
      }
      const int m_c = wu > 1 ? (5 * m_warm + 4 * wu - 1) / (4 * wu) : m_warm;
      uint32_t es, ec;
      top.bound2(m_warm, m_c, es, ec);
      if (lane == 0) {
        st.est[swarp] = es;
        st.est2[swarp] = ec;
      }
      Sel::sync();
      uint32_t ms = 0xFFFFFFFFu, mc = 0xFFFFFFFFu;
#pragma unroll
      for (int q = 0; q < kNS; ++q) {
        ms = min(ms, st.est[q]);
        mc = min(mc, st.est2[q]);
      }
      mk = ms;
      if (wu > 1 && mc > ms) {
        uint32_t c = top.count_ge(mc);
        const float flo = key_to_float(mc - 1u);  // key >= mc  <=>  value > flo
        for (int q = 1; q < wu; ++q) {
          const float* src;
          StageDesc d;
          uint32_t copied;
          stage_of(q, src, d, copied);
          if (copied == uint32_t(kUnit)) {
#pragma unroll 4
            for (int u = 0; u < kF4; ++u) {
              const float4 v = reinterpret_cast<const float4*>(src)[stt + kNST * u];
              c += (v.x > flo ? 1u : 0u) + (v.y > flo ? 1u : 0u) + (v.z > flo ? 1u : 0u) +
                   (v.w > flo ? 1u : 0u);
            }
          } else {
            for (int u = 0; u < kF4; ++u) {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const uint32_t pos = uint32_t(4 * (stt + kNST * u) + cc);
                float v = -__int_as_float(0x7F800000);
                if (pos < copied) v = src[pos];
                else if (pos < d.nvalid) v = __ldg(wrow + d.e0 + pos);
                c += v > flo ? 1u : 0u;
              }
            }
          }
        }
        c = __reduce_add_sync(0xFFFFFFFFu, c);
        if (lane == 0) atomicAdd(&st.warm_cnt, c);
        Sel::sync();
        if (st.warm_cnt >= uint32_t(k)) mk = mc;
      }
    }
  }
  mk = max(mk, mk_floor);
  if (stt == 0) {
    const uint64_t th0 = mk ? (uint64_t(mk) << 32) - 1ull : 0ull;
    if (th0) {
      // shared with the row's other CTAs without waiting for the reply (the
      // selector loop reads their thresholds back)
      if (pw.contributors > 1) atomicMax(&row_theta[pw.r], (unsigned long long)th0);
      atomicMax(&st.theta[w & 1], (unsigned long long)th0);
    }
    // A speculative threshold stays with this CTA (the row's other pieces
    // may adopt it as theirs, never as a proven bound); the row's end checks
    // it against the row's k-th word.
    if (spec > th0) {
      if (pw.contributors > 1) atomicMax(&row_spec[pw.r], (unsigned long long)spec);
      atomicMax(&st.theta[w & 1], (unsigned long long)spec);
      if (spec > st.spec[w & 1]) st.spec[w & 1] = spec;
    }
    __threadfence_block();
    atomicMax(&st.warm_pub, w + 1);
    TL_PIECE(w, 0);
  }
  Sel::sync();  // the bounds are read before the next warm start rewrites them
  return ok;
#undef wl
}

// The layer-20 block pool's block maxima, computed in the same pass (The
// Secret GPU Kernel Behind DeepSeek V4.1 Flash, video transcript 7:22-7:46):
// a block is eight consecutive positions, i.e. a filter thread's float4 and
// the next lane's; its score is the largest of its valid scores (NaN left
// out; NaN only when every valid score is NaN), +0.0 above -0.0.  Lanes with
// an even thread index store one float per block of the stage.
template <int T>
__device__ __forceinline__ void store_block_max(const float (&x)[kEPT], uint32_t valid, int ft,
                                                uint32_t e0, uint32_t nvalid, float* brow,
                                                int64_t bstride, uint32_t* status) {
  (void)bstride;
  (void)status;
  float bm[kF4];
  if (valid == 0xFFFFFFFFu) {  // a full unit: no element to leave out
#pragma unroll
    for (int u = 0; u < kF4; ++u) {
      const float m = fmaxf(fmaxf(x[4 * u], x[4 * u + 1]), fmaxf(x[4 * u + 2], x[4 * u + 3]));
      bm[u] = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));  // (fmaxf skips a NaN)
    }
  } else {
#pragma unroll
    for (int u = 0; u < kF4; ++u) {
      float v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        v[c] = ((valid >> (4 * u + c)) & 1u) ? x[4 * u + c] : __int_as_float(0x7FC00000);
      const float m = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      bm[u] = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    }
  }
  bool zero = false;
#pragma unroll
  for (int u = 0; u < kF4; ++u) zero |= bm[u] == 0.0f;
  if (__any_sync(0xFFFFFFFFu, zero)) {
    // a zero maximum: +0.0 if the block holds a valid +0.0, else -0.0
#pragma unroll
    for (int u = 0; u < kF4; ++u) {
      bool pz = false;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        pz |= ((valid >> (4 * u + c)) & 1u) && __float_as_uint(x[4 * u + c]) == 0u;
      pz |= __shfl_xor_sync(0xFFFFFFFFu, pz ? 1u : 0u, 1) != 0u;
      if (bm[u] == 0.0f) bm[u] = pz ? 0.0f : -0.0f;
    }
  }
  if ((ft & 1) == 0) {
    // block of the float4 pair (ft, ft + 1) in group u: (e0 + 4 ft) / 8 + (T / 2) u
    float* dst = brow + ((e0 + 4u * uint32_t(ft)) >> 3);
#pragma unroll
    for (int u = 0; u < kF4; ++u)
      if (uint32_t(4 * (ft + T * u)) < nvalid &&
          IN_BOUNDS(int64_t((e0 + 4u * uint32_t(ft)) >> 3) + (T / 2) * u < bstride, status))
        dst[(T / 2) * u] = bm[u];
  }
}

// ---------------------------------------------------------------------------
// The selection kernel.

__global__ void __launch_bounds__(kThreads, 1) topk_select_kernel(const Params p) {
  using Sel = Team<kNST, 1>;
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout sl = smem_layout(p.kp);
  float* ring = reinterpret_cast<float*>(smem + sl.ring);
  StageDesc* desc = reinterpret_cast<StageDesc*>(smem + sl.desc);
  uint64_t* const inbox0 = reinterpret_cast<uint64_t*>(smem + sl.inbox0);
  uint64_t* const inbox1 = reinterpret_cast<uint64_t*>(smem + sl.inbox1);
  uint64_t* tray = reinterpret_cast<uint64_t*>(smem + sl.tray);
  uint64_t* kept = reinterpret_cast<uint64_t*>(smem + sl.kept);
  uint32_t* perm = reinterpret_cast<uint32_t*>(smem + sl.perm);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + sl.hist);
  const int nstage = p.nstage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sl.bars);
  uint64_t* empty = full + nstage;
  __shared__ CtaState st;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int kp = p.kp, k = p.k;
  // (the wait limit is read from shared memory where it is used: a register
  // held across every role would cost the selector loop a spill)
#define wl (*reinterpret_cast<volatile uint32_t*>(&st.wait_limit))
  if (tid == 0) TL_SET(kTlStart, tl_now());
  // The next grid in the stream may be scheduled on SMs this one leaves; it
  // waits for this grid to complete before it reads global memory.
  if (tid == 0) grid_dep_launch();

  for (int j = tid; j < kp; j += kThreads) kept[j] = 0ull;
  for (int j = tid; j < kInbox; j += kThreads) {
    inbox0[j] = 0ull;
    inbox1[j] = 0ull;
  }
  if (tid == 0) {
    for (int q = 0; q < 2; ++q) {
      st.head[q] = 0;
      st.tail[q] = 0;
      st.fdone[q] = 0;
      st.theta[q] = 0ull;
      st.spec[q] = 0ull;
    }
    st.sel_pieces = 0;
    st.pieces_pub = 0;
    st.npieces = -1;
    st.warm_pub = 0;
    st.warm_claim = 0;
    st.first_issued = 0;
    st.fprog = 0u;
    st.flags = 0;
    st.wait_limit = p.wait_limit;
    for (int i = 0; i < nstage; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGW);  // the warps of the stage's filter group
    }
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) TL_SET(kTlSetup, tl_now());

  // ---------------- producer: the plan, a2 visiting orders, a3 copies ----------------
  if (warp == kProducerWarp) {
    const bool identity = (p.flags & TOPK_FLAG_IDENTITY_ORDER) != 0;
    // scores are read once: their lines go first when L2 needs room
    const uint64_t l2pol = l2_policy_evict_first();
    bool gave_up = false;
    bool stalled = false;  // test only: the producer stopped for good
    // Global memory (the plan's lengths and queue, the scores) only after the
    // grid before this one has completed.  The flat plan's pieces and
    // visiting orders are arithmetic: they are drawn before that wait.
    bool dep_done = false;
    auto dep_wait = [&]() {
      if (!dep_done) {
        grid_dep_wait();
        dep_done = true;
      }
    };
    if (p.plan != kPlanFlat) dep_wait();
    TL_CYC_DECL(tlc);
    uint32_t g = 0;  // stages issued (lane 0)
    int stage = 0;
    uint32_t phase = 0;
    int seq = 0;
    // wait for ring slot `stage` to be free, then hand it a descriptor
    auto next_slot = [&]() {
      TL_CLK(c0);
      if (g >= uint32_t(nstage) &&
          !mbar_wait_sleep(&empty[stage], phase ^ 1u, gave_up ? 1u : wl, 64))
        gave_up = true;
      TL_ACC(tlc, kCycProdWaitEmpty, c0);
    };
    auto advance = [&]() {
      ++g;
      if (++stage == nstage) {
        stage = 0;
        phase ^= 1u;
      }
    };
    for (int pi = 0;; ++pi) {
      Piece pc;
      bool bad_len;
      const int got = get_piece(p, pi, pc, bad_len);
      if (lane == 0 && pi == 0) TL_SET(kTlProdPiece, tl_now());
      if (lane == 0 && bad_len) atomicOr(p.status, TOPK_STATUS_BAD_LENGTH);
      if (got == 0) break;
      if (got == 2) continue;
      if (lane == 0) {
        // the descriptor slot is free once the selectors finished piece seq - kTable
        uint32_t it = gave_up ? wl : 0u;
        while (*reinterpret_cast<volatile int*>(&st.sel_pieces) < seq - kTable + 1) {
          if (++it > wl) {
            gave_up = true;
            break;
          }
          __nanosleep(256);
        }
        pc.g_first = g;  // the piece's first stage is the next one issued
        st.table[seq % kTable] = pc;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&st.pieces_pub) = seq + 1;
      }
      const float* row = p.scores + int64_t(pc.r) * p.row_stride;
      const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
      const int nu = pc.u_end - pc.u_begin;
      if (nu == 0 && lane == 0) {
        // an empty row still flows through the filters and selectors: one
        // stage with no elements
        dep_wait();
        next_slot();
        StageDesc d;
        d.e0 = 0;
        d.nvalid = 0;
        d.r = uint32_t(pc.r);
        d.tag = uint32_t(seq) | kFirst | kLast | kLastG;
        desc[stage] = d;
        mbar_arrive(&full[stage]);
        *reinterpret_cast<volatile int*>(&st.first_issued) = seq + 1;
        advance();
      }
      const int m_row = int((pc.L + kUnit - 1) / kUnit);
      const bool partial_tail = (pc.L % uint32_t(kUnit)) != 0;
      const int wu = warm_units(p.k, nu, pc.L);
      for (int c0 = 0; c0 < nu; c0 += kPermChunk) {
        const int cs = min(nu - c0, kPermChunk);
        // Full units first (the warm start reads the first wu units, its
        // bounds come from the first one): if the row's short last unit is
        // among them and the piece has more, swap it with the unit after
        // them; in a piece of at most wu units it is swapped to the end.
        const bool head_first = c0 == 0 && cs > wu;
        auto fix_head = [&]() {
          if (c0 == 0 && cs > 1 && partial_tail) {
            const int to = head_first ? wu : cs - 1;
            for (int q = 0; q < to; ++q) {
              if (pc.u_begin + int(perm[q] & uint32_t(kPermChunk - 1)) == m_row - 1) {
                const uint32_t t0 = perm[q];
                perm[q] = perm[to];
                perm[to] = t0;
              }
            }
          }
        };
        // lane 0: the copies of order positions [i0, i1) of this chunk
        auto issue = [&](int i0, int i1) {
          for (int i = i0; i < i1 && !stalled; ++i) {
            if (int64_t(g) == int64_t(p.stall_at)) {
              // test only: stop in front of this stage for good (its full
              // barrier never completes, so the waits behind it run out)
              stalled = true;
              break;
            }
            dep_wait();
            next_slot();
            const uint32_t u = uint32_t(pc.u_begin + c0) + (perm[i] & uint32_t(kPermChunk - 1));
            const uint32_t e0 = u * uint32_t(kUnit);
            const uint32_t nvalid = min(uint32_t(kUnit), pc.L - e0);
            const uint32_t bytes = aligned ? (nvalid & ~3u) * 4u : 0u;
            StageDesc d;
            d.e0 = e0;
            d.nvalid = nvalid;
            d.r = uint32_t(pc.r);
            d.tag = uint32_t(seq) | (c0 == 0 && i == 0 ? kFirst : 0u) |
                    (c0 + i == nu - 1 ? kLast : 0u) | (c0 + i >= nu - 2 ? kLastG : 0u);
            desc[stage] = d;
            fence_proxy_async_smem();
            if (bytes) {
              mbar_arrive_expect_tx(&full[stage], bytes);
              bulk_load_hint(ring + stage * kUnit, row + e0, bytes, &full[stage], l2pol);
            } else {
              mbar_arrive(&full[stage]);
            }
            if (g == 0u) TL_SET(kTlFirstCopy, tl_now());
            // Until a piece's first wu stages are issued, their ring slots'
            // barriers may still be in an earlier phase: the selectors look at
            // them only after this count says the stages are on their way.
            if (c0 + i == wu - 1) *reinterpret_cast<volatile int*>(&st.first_issued) = seq + 1;
            if (c0 + i == nu - 1) TL_PIECE(seq, 13);
            advance();
          }
        };
        // The piece's first units are the smallest keys of its first chunk:
        // for chunks of up to 64 units their copies go out (phase 0) before
        // the rest of the order is sorted (phase 1).
        const bool early = head_first && cs <= 64;
        for (int ph = early ? 0 : 1; ph < 2 && !stalled; ++ph) {
          if (ph == 0) {
            visit_order_head(perm, cs, int64_t(pc.u_begin) + c0, pc.r, p.seed_lo, p.seed_hi,
                             identity, lane, wu + 1);
          } else {
            build_visit_order_warp(perm, cs, int64_t(pc.u_begin) + c0, pc.r, p.seed_lo,
                                   p.seed_hi, identity, lane);
            if (lane == 0 && seq == 0 && c0 == 0) TL_SET(kTlProdOrder, tl_now());
          }
          if (lane == 0) {
            fix_head();
            issue(ph == 0 ? 0 : (early ? wu : 0), ph == 0 ? wu : cs);
          }
          __syncwarp();
          stalled = __shfl_sync(0xFFFFFFFFu, stalled, 0);
        }
        __syncwarp();  // the order buffer is reused by the next chunk
        stalled = __shfl_sync(0xFFFFFFFFu, stalled, 0);
        if (stalled) break;
      }
      ++seq;
      if (stalled) break;
    }
    dep_wait();
    if (lane == 0) {
      TL_SET(kTlLastCopy, tl_now());
      *reinterpret_cast<volatile int*>(&st.npieces) = seq;
      // the copies of the last stages have landed before this warp (and so
      // the CTA) can leave, even if the filters gave up on them
      for (uint32_t q = g > uint32_t(nstage) ? g - uint32_t(nstage) : 0u; q < g; ++q)
        if (!mbar_wait(&full[q % uint32_t(nstage)], (q / uint32_t(nstage)) & 1u, wl))
          gave_up = true;
      if (stalled) return;  // (test only: no end marker either)
      // one end marker for each filter group (consecutive stages alternate)
      for (int q = 0; q < kFG; ++q) {
        next_slot();
        StageDesc d;
        d.e0 = 0;
        d.nvalid = 0;
        d.r = 0;
        d.tag = kEnd;
        desc[stage] = d;
        mbar_arrive(&full[stage]);
        advance();
      }
      if (gave_up) atomicOr(p.status, TOPK_STATUS_TIMEOUT);
      TL_FLUSH(tlc);
      TL_SET(kTlInfo, (unsigned long long)smid() | ((unsigned long long)seq << 32));
      TL_SET(kTlProdExit, tl_now());
    }
    return;
  }

  // ---------------- filter warps: a4 + a5 ----------------
  // Two groups of kGW warps take alternate ring stages (group q the stages
  // g = q, q + 2, ...); a group's 128 threads test a whole 8192-element unit,
  // 64 elements a thread as two contiguous 4096-element halves.  A warp thus
  // pays a stage's fixed costs (the wait, the descriptor, the release, and the
  // candidate path when some lane has a survivor) once for 2048 elements, and
  // the two groups' latencies overlap.
  if (warp < kNF) {
    grid_dep_wait();  // (before any global access: see the producer)
    const int grp = warp / kGW;     // filter group
    const int tg = tid - grp * kGT;  // 0 .. kGT-1 within the group
    uint64_t th = 0ull;
    float thf = threshold_float(th);
    uint32_t admitted = 0;
    bool saw_nan = false, timed_out = false;
    uint32_t gs = uint32_t(grp);  // global index of the group's next stage
    int cur_seq = -1;             // piece of the stages seen last
    int par = 0;
    int32_t r = 0;
    const bool tl0 = tid == 0;  // (timeline: filter warp 0, lane 0)
    TL_CYC_DECL(tlc);
    (void)tl0;
    const float* row = p.scores;
    bool aligned = true;
    // every exit decision is warp-uniform: a wait that gave up in any lane
    // ends the warp's loop
    for (;;) {
      const int stage = int(gs % uint32_t(nstage));
      const uint32_t phase = (gs / uint32_t(nstage)) & 1u;
      TL_CLK(cw);
      if (!mbar_wait_sleep(&full[stage], phase, wl, 32)) timed_out = true;
      if (tl0) TL_ACC(tlc, kCycFiltWaitFull, cw);
      TL_CLK(cbody);
      const StageDesc d = desc[stage];
      if (__any_sync(0xFFFFFFFFu, timed_out)) {
        timed_out = true;
        break;
      }
      if (d.tag & kEnd) break;
      const int seq = int(d.tag & kSeqMask);
      if (seq != cur_seq) {
        // The group's first stage of a piece: wait for its starting
        // threshold (see filter_wait_theta).
        cur_seq = seq;
        par = seq & 1;
        TL_CLK(ct);
        if (lane == 0 && !filter_wait_theta(p.row_theta, p.row_spec, st, seq, wl)) timed_out = true;
        if (__any_sync(0xFFFFFFFFu, timed_out)) {
          timed_out = true;
          break;
        }
        if (tl0) {
          TL_ACC(tlc, kCycFiltWaitTheta, ct);
          if (seq == 0) TL_SET(kTlFiltFirst, tl_now());
          TL_PIECE(seq, 1);
        }
        r = int32_t(d.r);
        row = p.scores + int64_t(r) * p.row_stride;
        aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
        th = *reinterpret_cast<volatile unsigned long long*>(&st.theta[par]);
        thf = threshold_float(th);
      } else {
        const uint64_t nt = *reinterpret_cast<volatile unsigned long long*>(&st.theta[par]);
        if (nt != th) {
          th = nt;
          thf = threshold_float(th);
        }
      }
      const float* src = ring + stage * kUnit;
      const uint32_t e0 = d.e0, nvalid = d.nvalid;
      const uint32_t copied = aligned ? (nvalid & ~3u) : 0u;
      // Most stages have no element past the threshold: the test first folds
      // each float4 group into one bit (a superset: it also passes NaN, ties
      // and padding); only flagged groups are re-read (where they sit: the
      // stage is not released yet, or past the copied prefix of a ragged
      // unit, global memory) and classified element by element.  Group ug
      // (0 .. 15) of this thread is float4 tg + kGT ug of the unit.
      uint32_t gm = 0;
      uint64_t valid = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t hb = uint32_t(h) * uint32_t(kUnit / 2);
        const uint32_t nv_h = nvalid > hb ? min(nvalid - hb, uint32_t(kUnit / 2)) : 0u;
        const uint32_t cp_h = copied > hb ? min(copied - hb, uint32_t(kUnit / 2)) : 0u;
        float x[kEPT];
        const uint32_t vh = load_share<kGT>(x, src + hb, row, e0 + hb, nv_h, cp_h, tg);
        if (p.bmax != nullptr)
          store_block_max<kGT>(x, vh, tg, e0 + hb, nv_h, p.bmax + int64_t(r) * p.bstride,
                               p.bstride, p.status);
        valid |= uint64_t(vh) << (32 * h);
#pragma unroll
        for (int u = 0; u < kF4; ++u)
          gm |= uint32_t(!(x[4 * u + 0] < thf) | !(x[4 * u + 1] < thf) | !(x[4 * u + 2] < thf) |
                         !(x[4 * u + 3] < thf)) << (u + kF4 * h);
      }
      // element e (0 .. 63) of this thread: unit position 4 (tg + kGT (e / 4)) + e % 4
      auto pos_of = [&](int e) -> uint32_t {
        return uint32_t(4 * (tg + kGT * (e >> 2)) + (e & 3));
      };
      auto word_of = [&](uint32_t bits, int e) -> uint64_t {
        return (uint64_t(order_key(bits)) << 32) | uint64_t(~(e0 + pos_of(e)));
      };
      auto elem_bits = [&](int e) -> uint32_t {
        const uint32_t pos = pos_of(e);
        if (pos < copied) return __float_as_uint(src[pos]);
        return __float_as_uint(__ldg(row + e0 + pos));
      };
      if (tl0) TL_CNT(tlc, kCycFiltStages);
      if (tl0) TL_ACC(tlc, kCycFiltLoad, cbody);
      TL_CLK(cc);
      if (__any_sync(0xFFFFFFFFu, gm != 0u)) {
        if (tl0) TL_CNT(tlc, kCycFiltCandStages);
        // the inbox head as of now (it only grows: a safe bound for the room
        // check below, read early so its latency overlaps the classification)
        const uint32_t head_seen = *reinterpret_cast<volatile uint32_t*>(&st.head[par]);
        // A strict float compare is already the exact word test for every
        // value except NaN and values equal to the threshold's own (ties,
        // and -0.0 against +0.0): those few get the 64-bit word test.
        TL_CLK(ccl);
        uint64_t passm = 0;
        for (uint32_t gg = gm; gg; gg &= gg - 1u) {
          const int ug = __ffs(gg) - 1;
          float4 v;
          if (copied == uint32_t(kUnit)) {
            v = reinterpret_cast<const float4*>(src)[tg + kGT * ug];
          } else {
            v.x = __uint_as_float(((valid >> (4 * ug + 0)) & 1u) ? elem_bits(4 * ug + 0) : 0u);
            v.y = __uint_as_float(((valid >> (4 * ug + 1)) & 1u) ? elem_bits(4 * ug + 1) : 0u);
            v.z = __uint_as_float(((valid >> (4 * ug + 2)) & 1u) ? elem_bits(4 * ug + 2) : 0u);
            v.w = __uint_as_float(((valid >> (4 * ug + 3)) & 1u) ? elem_bits(4 * ug + 3) : 0u);
          }
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int e = 4 * ug + c;
            bool pass = vv[c] > thf;
            if (!(vv[c] < thf) && !pass) {  // equal to the threshold's value, or NaN
              const uint32_t bits = __float_as_uint(vv[c]);
              const bool nan = (bits & 0x7FFFFFFFu) > 0x7F800000u;
              saw_nan |= nan && ((valid >> e) & 1u);
              pass = !nan && word_of(bits, e) > th;
            }
            passm |= uint64_t(pass) << e;
          }
        }
        passm &= valid;
        const uint32_t np = uint32_t(__popcll(passm));
#if TL_CYCLES
        __syncwarp();
        if (tl0) TL_ACC(tlc, kCycCandClassify, ccl);
        const long long cres = clock64();
        const unsigned long long tl_words = __reduce_add_sync(0xFFFFFFFFu, np);
        if (tl0) tlc[kCycCandWords] += tl_words;
#endif
        if (np) {
          uint32_t pos = atomicAdd(&st.tail[par], np);
          admitted += np;
          // wait for room: the selectors free slots by advancing head (the
          // head seen at the stage's start usually shows room already)
          if (pos + np - head_seen > uint32_t(kInbox)) {
            uint32_t it = timed_out ? wl : 0u;
            while (pos + np - *reinterpret_cast<volatile uint32_t*>(&st.head[par]) >
                   uint32_t(kInbox)) {
              if (++it > wl) {
                timed_out = true;
                break;
              }
              __nanosleep(64);
            }
          }
#if TL_CYCLES
          if (tl0) TL_ACC(tlc, kCycCandReserve, cres);
#endif
          volatile uint64_t* ib = par ? inbox1 : inbox0;
          for (uint64_t mm = passm; mm; mm &= mm - 1ull) {
            const int e = __ffsll(mm) - 1;
            ib[pos & (kInbox - 1)] = word_of(elem_bits(e), e);
            ++pos;
          }
        }
#if TL_CYCLES
        __syncwarp();
        if (tl0) TL_ACC(tlc, kCycCandWrite, cres);
#endif
      }
      if (tl0) TL_ACC(tlc, kCycFiltCand, cc);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[stage]);
        // (the selectors' pre-final compares this with global stage indices)
        if (warp == 0) *reinterpret_cast<volatile uint32_t*>(&st.fprog) = gs + 1u;
      }
      if (tl0) TL_ACC(tlc, kCycFiltBody, cbody);
      if (lane == 0 && (d.tag & kLastG) && (tid == 0 || tid == kGT)) TL_PIECE(seq, tid == 0 ? 2 : 12);
      // every warp reports each stage it has finished (its words reserved):
      // the selectors know how many stages a piece has
      __syncwarp();
      if (d.tag & kLastG) {
        // the group's last stage of the piece: its admitted count
        admitted = __reduce_add_sync(0xFFFFFFFFu, admitted);
        if (lane == 0 && admitted) atomicAdd(&p.admitted[r], admitted);
        admitted = 0;
      }
      if (lane == 0) {
        __threadfence_block();
        atomicAdd(&st.fdone[par], 1);
      }
      gs += uint32_t(kFG);
    }
    saw_nan = __any_sync(0xFFFFFFFFu, saw_nan);
    timed_out = __any_sync(0xFFFFFFFFu, timed_out);
    if (lane == 0) {
      if (saw_nan) atomicOr(p.status, TOPK_STATUS_NAN);
      if (timed_out) atomicOr(p.status, TOPK_STATUS_TIMEOUT);
    }
    if (tl0) {
      TL_FLUSH(tlc);
      TL_SET(kTlFiltExit, tl_now());
    }
    return;
  }

  // ---------------- selector warps: a6, a7, a8 ----------------
  grid_dep_wait();  // (before any global access: see the producer)
  const int stt = tid - kNFT;  // 0 .. kNST-1
  const int swarp = stt >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  bool timed_out = false;
  uint32_t nsorts = 0, nsorted = 0;
  int tray_n = 0;       // words in the tray
  int kept_n = 0;       // real words in the kept list
  int pruned = 0;       // tray words left by the last prune
  uint64_t theta = 0ull;         // the piece's threshold word (proven or speculative)
  uint64_t theta_proven = 0ull;  // the largest proven word this piece has published
  uint32_t head = 0, head_other = 0;  // inbox heads: this piece's parity, the other one
  int par = 0;
  int warm_next = 0;  // next piece whose starting threshold is to be set
  int fd_cum0 = 0, fd_cum1 = 0;  // filter completions expected so far, per inbox parity
  TL_CYC_DECL(tlc);   // (timeline: accumulated by selector thread 0)

  // Publish a threshold to the filters (and to the row's other CTAs).
  // Every word passed here is proven: at least k words of the row are at or
  // above it.  (The threshold word the filters use may also hold a
  // speculative start, which is never shared as a proven bound.)
  auto raise_theta = [&](uint64_t nth, const Piece& pc) {
    if (nth > theta_proven) {
      theta_proven = nth;
      // shared with the row's other CTAs without waiting for the reply (the
      // selector loop reads their thresholds back)
      if (stt == 0 && pc.contributors > 1) atomicMax(&p.row_theta[pc.r], (unsigned long long)nth);
    }
    if (nth <= theta) return;
    theta = nth;
    if (stt == 0) atomicMax(&st.theta[par], (unsigned long long)nth);
  };

  // a6: the tray.  A byte-wise histogram select over kept + tray finds a word
  // prefix T such that at least k words are >= T and at most kp + slack are;
  // tray words below T can never reach the best k and are dropped, and the
  // threshold rises to T.  With `sort` (the tray has passed its mark, or the
  // piece is done) the rest are bitonic-sorted and merged into the kept
  // list, whose k-th word becomes the threshold, and the tray is emptied.
  auto process_tray = [&](bool sort, bool final, const Piece& pc) {
    // at the end of a piece the select is exact (no slack): at most kp words
    // are left to sort
    const int slack = (final || kp >= kTrayMark) ? 0 : kSelectSlack;
    uint64_t T = 0ull;
    if (kept_n + tray_n > kp + slack) {
      uint64_t prefix = 0ull;
      uint32_t need = uint32_t(k), greater = 0;
      for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        const uint64_t hmask = pass == 0 ? 0ull : (~0ull << (shift + 8));
        for (int b = stt; b < 256; b += kNST) hist[b] = 0u;
        Sel::sync();
        // the kept list holds its kept_n real words first
        const int nw = kept_n + tray_n;
        for (int j = stt; j < nw; j += kNST) {
          const uint64_t w = j < kept_n ? kept[j] : tray[j - kept_n];
          if ((w & hmask) == prefix) atomicAdd(&hist[uint32_t(w >> shift) & 0xFFu], 1u);
        }
        Sel::sync();
        if (swarp == 0) {
          // lane l owns bins 255-8l .. 248-8l, scanned from the top
          uint32_t cnt8[8], sum = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            cnt8[q] = hist[255 - 8 * lane - q];
            sum += cnt8[q];
          }
          uint32_t incl = sum;
#pragma unroll
          for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += o;
          }
          const uint32_t excl = incl - sum;
          if (excl < need && incl >= need) {
            uint32_t acc = excl;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (acc < need && acc + cnt8[q] >= need) {
                st.sel_b = 255 - 8 * lane - q;
                st.sel_above = int(acc);
                st.sel_binc = int(cnt8[q]);
              }
              acc += cnt8[q];
            }
          }
        }
        Sel::sync();
        const uint32_t b = uint32_t(st.sel_b);
        const uint32_t above = uint32_t(st.sel_above), binc = uint32_t(st.sel_binc);
        prefix |= uint64_t(b) << shift;
        greater += above;
        need -= above;
        // a prune stops at a 16-bit key prefix: a bound, not the exact word
        if (greater + binc <= uint32_t(kp + slack) || pass == 7 || (!sort && pass == 1)) {
          T = prefix;
          break;
        }
      }
    }
    // keep the tray words >= T, compacting in rounds that never overwrite a
    // word not yet read (a kept word only moves to a lower position)
    if (stt == 0) st.cnt2 = 0;
    Sel::sync();
    constexpr int R = 8;
    for (int base0 = 0; base0 < tray_n; base0 += R * kNST) {
      uint64_t w[R];
      bool keep[R];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const int t = base0 + u * kNST + stt;
        w[u] = t < tray_n ? tray[t] : 0ull;
        keep[u] = w[u] != 0ull && w[u] >= T;
      }
      Sel::sync();
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, keep[u]);
        if (mask) {
          int at = 0;
          if (lane == 0) at = atomicAdd(&st.cnt2, __popc(mask));
          at = __shfl_sync(0xFFFFFFFFu, at, 0);
          if (keep[u] && IN_BOUNDS(at + __popc(mask & lt_mask) < kTray, p.status))
            tray[at + __popc(mask & lt_mask)] = w[u];
        }
      }
    }
    Sel::sync();
    const int r = st.cnt2;
    if (!sort) {
      tray_n = r;
      pruned = r;
      raise_theta(T ? T - 1ull : 0ull, pc);
      return;
    }
    // the bitonic tray sort: sort the r survivors (padded with empty words
    // to a power of two, at least one word per selector thread) and merge
    // them in
    const int P = max(next_pow2_dev(max(r, 1)), kNST);
    if (!IN_BOUNDS(P <= kTray, p.status)) return;
    for (int t = r + stt; t < P; t += kNST) tray[t] = 0ull;
    Sel::sync();
    team_sort_desc<Sel>(tray, P, 2, stt);
    if (kept_n == 0) {
      // nothing kept yet: the sorted tray is the list
      for (int q = stt; q < kp; q += kNST) kept[q] = q < P ? tray[q] : 0ull;
      Sel::sync();
    } else {
      merge_into_kept<Sel>(kept, tray, P, kp, stt);
    }
    ++nsorts;
    nsorted += uint32_t(r);
    kept_n = min(kp, kept_n + r);
    tray_n = 0;
    pruned = 0;
    raise_theta(kept[k - 1], pc);
  };

  // Move `n` reserved words of inbox `par` into the tray (a slot still 0 is
  // reserved but not yet written: wait for it), and free their slots.
  auto take = [&](int n) {
    volatile uint64_t* ib = par ? inbox1 : inbox0;
    const uint32_t h = head;
    for (int j = stt; j < n; j += kNST) {
      volatile uint64_t* slot = ib + ((h + uint32_t(j)) & (kInbox - 1));
      uint64_t w = *slot;
      uint32_t it = timed_out ? wl : 0u;
      while (w == 0ull) {
        if (++it > wl) {
          timed_out = true;
          break;
        }
        __nanosleep(32);
        w = *slot;
      }
      *slot = 0ull;
      if (IN_BOUNDS(tray_n + j < kTray, p.status)) tray[tray_n + j] = w;
    }
    __threadfence_block();  // the emptied slots are visible before head moves
    Sel::sync();
    head = h + uint32_t(n);
    tray_n += n;
    if (stt == 0) *reinterpret_cast<volatile uint32_t*>(&st.head[par]) = head;
  };

  // A row whose speculative start missed (fewer than k of its words lie above
  // the largest speculative threshold its pieces started from) is selected
  // again, exactly, by this team alone from global memory: every word of the
  // row at or above `lb` goes through the tray into a fresh kept list.  `lb`
  // is a word the row's k-th word is known to reach (a word of the row's
  // merged or kept list), or 0.
  auto rescan = [&](const Piece& pc, uint64_t lb) {
    const float* rrow = p.scores + int64_t(pc.r) * p.row_stride;
    for (int q = stt; q < kp; q += kNST) kept[q] = 0ull;
    kept_n = 0;
    tray_n = 0;
    pruned = 0;
    theta = lb ? lb - 1ull : 0ull;
    if (stt == 0) atomicOr(p.status, TOPK_STATUS_RESCAN);
    Sel::sync();
    constexpr int R = kRescanChunk / kNST;
    static_assert(kRescanChunk % kNST == 0 && kTray >= 2 * kRescanChunk - 1024,
                  "a rescan step fits the tray after a sort");
    for (uint32_t b0 = 0; b0 < pc.L; b0 += uint32_t(kRescanChunk)) {
      if (tray_n + kRescanChunk > kTray) process_tray(true, false, pc);
      if (stt == 0) st.cnt2 = 0;
      Sel::sync();
      uint32_t bits[R];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const uint32_t e = b0 + uint32_t(u * kNST + stt);
        bits[u] = e < pc.L ? __float_as_uint(rrow[e]) : 0x7FFFFFFFu;  // (past the end: a NaN)
      }
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const uint32_t e = b0 + uint32_t(u * kNST + stt);
        const uint64_t w = (uint64_t(order_key(bits[u])) << 32) | uint64_t(~e);
        const bool keep = (bits[u] & 0x7FFFFFFFu) <= 0x7F800000u && w > theta;  // NaN never
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, keep);
        if (mask) {
          int at = 0;
          if (lane == 0) at = atomicAdd(&st.cnt2, __popc(mask));
          at = __shfl_sync(0xFFFFFFFFu, at, 0);
          if (keep && IN_BOUNDS(tray_n + at + __popc(mask & lt_mask) < kTray, p.status))
            tray[tray_n + at + __popc(mask & lt_mask)] = w;
        }
      }
      Sel::sync();
      tray_n += st.cnt2;
      Sel::sync();
    }
    if (tray_n > 0) process_tray(true, true, pc);
  };

  for (int j = 0;; ++j) {
    // the producer publishes piece j's descriptor before its first stage
    if (stt == 0) {
      uint32_t it = timed_out ? wl : 0u;
      int have = 0;
      for (;;) {
        if (*reinterpret_cast<volatile int*>(&st.pieces_pub) > j) {
          have = 1;
          break;
        }
        if (*reinterpret_cast<volatile int*>(&st.npieces) >= 0) {
          have = *reinterpret_cast<volatile int*>(&st.pieces_pub) > j ? 1 : 0;
          break;
        }
        if (++it > wl) {
          timed_out = true;
          break;
        }
        __nanosleep(128);
      }
      st.flags = have;
    }
    Sel::sync();
    const bool have = st.flags != 0;
    const Piece pc = st.table[j % kTable];
    Sel::sync();
    if (!have) break;
    par = j & 1;
    if (j > 0) {  // pieces alternate inboxes: pick up this parity's head
      const uint32_t h = head;
      head = head_other;
      head_other = h;
    }
    const int pc_nu = pc.u_end - pc.u_begin;
    // stage reports that make the piece done: every warp of a stage's group
    // reports it (an empty row is one stage), added up per inbox parity
    const int fd_add = kGW * max(pc_nu, 1);
    if (par) fd_cum1 += fd_add;
    else fd_cum0 += fd_add;
    const int fd_target = par ? fd_cum1 : fd_cum0;
    const uint32_t pre_at = pc.g_first + uint32_t(pc_nu) - uint32_t(kPreFinal);
    bool pre_done = pc_nu < kPreFinalMin;

    for (;;) {
      // One lane polls until there is a batch to take or the piece is done;
      // the rest of the team waits at the barrier.  The finished-filter count
      // is read before the tail, so a full count means the tail is final.
      TL_CLK(cpoll);
      if (stt == 0) {
        uint32_t it = timed_out ? wl : 0u;
        int n = 0, done = 0, warm = 0, pre = 0;
        for (;;) {
          // First: a piece (this one or the next) still waiting for its
          // starting threshold.  A split row whose other CTAs have already
          // published a threshold starts from that one at once (action 2);
          // otherwise the warm start runs once its units have landed
          // (action 1).  Either is claimed first: the filters may already
          // have taken the piece on (they adopt a split row's shared
          // threshold when they reach the piece first): then it is skipped
          // (action 3).
          bool warm_due = false;
          if (warm_next <= j + 1 && *reinterpret_cast<volatile int*>(&st.warm_claim) > warm_next) {
            warm = 3;
            break;
          }
          if (warm_next <= j + 1 && *reinterpret_cast<volatile int*>(&st.pieces_pub) > warm_next) {
            const Piece& pn = st.table[warm_next % kTable];
            const unsigned long long rt =
                pn.contributors > 1
                    ? *reinterpret_cast<volatile unsigned long long*>(&p.row_theta[pn.r])
                    : 0ull;
            // a speculative start of the row's other pieces is adopted as
            // this piece's own (the row's end checks the largest of them)
            const unsigned long long rs =
                pn.contributors > 1
                    ? *reinterpret_cast<volatile unsigned long long*>(&p.row_spec[pn.r])
                    : 0ull;
            if (rt != 0ull || rs != 0ull) {
              warm = 3;
              if (atomicCAS(&st.warm_claim, warm_next, warm_next + 1) == warm_next) {
                adopt_row_theta(st, warm_next, rt, rs);
                warm = 2;
              }
              break;
            }
            if (*reinterpret_cast<volatile int*>(&st.first_issued) > warm_next) {
              // Copies can land out of order: for the next piece every
              // warm-start unit must be in (the warm start must not block
              // while this piece's inbox still needs draining).  For the
              // current piece the filters have finished everything before
              // it, so the producer can land the remaining units while the
              // warm start works on the first one: it starts once that one
              // is in.
              const int wu = warm_units(k, pn.u_end - pn.u_begin, pn.L);
              const int need = warm_next == j ? 1 : wu;
              bool landed = true;
              for (int q = 0; q < need && landed; ++q) {
                const uint32_t g = pn.g_first + uint32_t(q);
                landed = mbar_try_wait(&full[g % uint32_t(nstage)], (g / uint32_t(nstage)) & 1u);
              }
              if (landed) {
                warm = atomicCAS(&st.warm_claim, warm_next, warm_next + 1) == warm_next ? 1 : 3;
                break;
              }
              warm_due = true;  // issued, not landed yet
            }
          }
          const int fd = *reinterpret_cast<volatile int*>(&st.fdone[par]);
          const uint32_t tail = *reinterpret_cast<volatile uint32_t*>(&st.tail[par]);
          const uint32_t avail = tail - head;
          n = int(min(avail, uint32_t(kTray - tray_n)));
          if (n > kTakeMax) n = kTakeMax;
          if (fd < fd_target && avail < uint32_t(kTakeMin)) n = 0;
          done = (fd >= fd_target && avail == 0) ? 1 : 0;
          // the filters wait on the next piece's threshold, not on this
          // piece's end: a warm start whose units are on their way goes first
          if (done && warm_due) done = 0;
          // (the row's shared word is in global memory: an L2 round trip,
          // so it is looked at on every fourth poll only)
          if (pc.contributors > 1 && (it & 3u) == 0u) {
            const unsigned long long gt =
                *reinterpret_cast<volatile unsigned long long*>(&p.row_theta[pc.r]);
            if (gt > theta) atomicMax(&st.theta[par], gt);
          }
          // near the piece's end: take everything there is and sort it
          if (!pre_done && !done &&
              int32_t(*reinterpret_cast<volatile uint32_t*>(&st.fprog) - pre_at) >= 0) {
            pre = 1;
            n = int(min(avail, uint32_t(kTray - tray_n)));
            if (n > kTakeMax) n = kTakeMax;
            break;
          }
          if (n > 0 || done) break;
          if (++it > wl) {
            timed_out = true;
            done = 1;
            break;
          }
          __nanosleep(256);
        }
        st.sel_n = n;
        st.sel_done = done;
        st.flags = warm;
        st.sel_pre = pre;
      }
      Sel::sync();
      const int n = st.sel_n;
      const bool done = st.sel_done != 0;
      const int warm = st.flags;
      const bool pre = st.sel_pre != 0;
      const uint64_t sth = *reinterpret_cast<volatile unsigned long long*>(&st.theta[par]);
      if (sth > theta) theta = sth;
      Sel::sync();
      if (stt == 0) TL_ACC(tlc, kCycSelPoll, cpoll);
      if (warm) {
        TL_CLK(cw);
        if (warm == 1 && !warm_start_piece(p.scores, p.row_stride, p.row_theta, p.row_spec, st,
                                           warm_next, ring, desc, full, nstage, k, stt))
          timed_out = true;
        if (stt == 0) TL_ACC(tlc, kCycSelWarm, cw);
        ++warm_next;
        continue;
      }
      if (pre) {
        pre_done = true;
        if (stt == 0) TL_PIECE(j, 9);
        TL_CLK(ct);
        if (n > 0) take(n);
        if (stt == 0) TL_ACC(tlc, kCycSelTake, ct);
        TL_CLK(cs);
        if (tray_n > 0) process_tray(true, true, pc);
        if (stt == 0) TL_ACC(tlc, kCycSelSort, cs);
        if (stt == 0) TL_PIECE(j, 7);
        continue;
      }
      if (done) break;
      TL_CLK(ct);
      take(n);
      if (stt == 0) TL_ACC(tlc, kCycSelTake, ct);
      TL_CLK(cs);
      if (tray_n >= kTrayMark) {
        process_tray(true, false, pc);
        if (stt == 0) TL_ACC(tlc, kCycSelSort, cs);
      } else if (tray_n >= pruned + kPruneStep) {
        process_tray(false, false, pc);
        if (stt == 0) TL_ACC(tlc, kCycSelPrune, cs);
      }
    }

    // end of the piece: final sort, then the row's output (directly, or
    // through the split-row ticket)
    TL_CLK(cend);
    if (stt == 0) TL_PIECE(j, 8);
    if (tray_n > 0) {
      if (tray_n <= kp && kp >= kNST) {
        // At most kp words are left (the kept list, if any, holds the best kp
        // of everything before): sort them and merge them in, or take them
        // as the list -- no select needed.
        const int P = max(next_pow2_dev(tray_n), kNST);  // <= kp
        for (int t = tray_n + stt; t < P; t += kNST) tray[t] = 0ull;
        Sel::sync();
        team_sort_desc<Sel>(tray, P, 2, stt);
        if (stt == 0) TL_PIECE(j, 10);
        if (kept_n > 0) {
          merge_into_kept<Sel>(kept, tray, P, kp, stt);
        } else {
          for (int q = stt; q < kp; q += kNST) kept[q] = q < P ? tray[q] : 0ull;
          Sel::sync();
        }
        ++nsorts;
        nsorted += uint32_t(tray_n);
        kept_n = min(kp, kept_n + tray_n);
        tray_n = 0;
      } else {
        process_tray(true, true, pc);
      }
    }
    if (stt == 0) TL_PIECE(j, 4);
    // A row whose pieces started from speculative thresholds is selected
    // again if its k-th word does not lie above the largest of them.
    bool redo = false;
    uint64_t redo_lb = 0ull;
    if (stt == 0) {
      atomicAdd(&p.sorts[pc.r], nsorts);
      atomicAdd(&p.survivors[pc.r], nsorted);
    }
    nsorts = 0;
    nsorted = 0;
    if (pc.contributors == 1) {
      const uint64_t spec_p = st.spec[par];
      if (spec_p != 0ull && kept[k - 1] <= spec_p) {
        redo = true;
        redo_lb = kept[k - 1];
      } else {
        write_row(p, pc.r, kept, stt, kNST);
      }
    } else {
      // a7: publish the local list, take a ticket; the last ticket merges.
      uint64_t* mine = p.partials + int64_t(pc.slot) * kp;
      if (IN_BOUNDS(pc.slot >= 0 && pc.slot < p.nslots, p.status))
        for (int q = stt; q < kp; q += kNST) mine[q] = kept[q];
      __threadfence();
      Sel::sync();
      if (stt == 0) {
        TL_PIECE(j, 11);
        const uint32_t t = atomicAdd(&p.tickets[pc.r], 1u);
        st.leader = (t == uint32_t(pc.contributors - 1)) ? 1 : 0;
        TL_PIECE(j, 5);
      }
      Sel::sync();
      if (st.leader) {
        if (stt == 0) TL_CNT(tlc, kCycSelLeader);
        __threadfence();
        // (read now, used after the merge: the row's pieces all published
        // their speculative words before their tickets)
        const uint64_t rs = *reinterpret_cast<volatile unsigned long long*>(&p.row_spec[pc.r]);
        // Gather lists into this piece's (drained) inbox + the tray and merge
        // them as a tree of parallel pairwise merges; the running result
        // stays in slot 0.
        uint64_t* slots = par == 0 ? inbox0 : tray;  // kInbox + kTray contiguous words
        const int cap = (kInbox + kTray) / kp;
        const int lkp = __ffs(kp) - 1;
        for (int q = stt; q < kp; q += kNST) slots[q] = kept[q];
        int gathered = 0;  // other contributors gathered so far (never this CTA)
        int remaining = pc.contributors - 1;
        while (remaining > 0) {
          const int takeq = min(remaining, min(cap - 1, 16));
          if (stt < takeq) {
            const int i = gathered + stt;
            const int o = i + (i >= pc.self ? 1 : 0);  // contributor index
            int64_t slot;
            if (p.plan != kPlanFlat) {  // items or queue: slot r * split + segment
              slot = int64_t(pc.r) * p.split + o;
            } else {
              const int64_t M = int64_t(p.rows) * p.u_full, G = gridDim.x;
              const int64_t go = pc.first_cta + o;
              slot = 2 * go + (udiv(flat_lo(go, M, G), p.u_full) == pc.r ? 0 : 1);
            }
            if (!IN_BOUNDS(slot >= 0 && slot < p.nslots, p.status)) slot = 0;
            st.gsrc[stt] = p.partials + slot * kp;
          }
          Sel::sync();
          // every word of the step with eight loads in flight per thread
          const int total = takeq * kp;
          for (int b = stt; b < total; b += 8 * kNST) {
            uint64_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int t = b + u * kNST;
              v[u] = t < total ? __ldcg(st.gsrc[t >> lkp] + (t & (kp - 1))) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int t = b + u * kNST;
              if (t < total && IN_BOUNDS(kp + t < kInbox + kTray, p.status)) slots[kp + t] = v[u];
            }
          }
          gathered += takeq;
          remaining -= takeq;
          Sel::sync();
          const int nl = takeq + 1;
          for (int gap = 1; gap < nl; gap <<= 1) {
            // pairs (q, q + gap) for q a multiple of 2*gap with q + gap < nl
            const int npairs = (nl - gap + 2 * gap - 1) / (2 * gap);
            for (int u = stt; u < npairs * kp; u += kNST) {
              const int pr = u / kp, q = u - pr * kp;
              uint64_t* a = slots + (2 * gap * pr) * kp;
              const uint64_t* b = a + gap * kp;
              const uint64_t x = a[q], y = b[kp - 1 - q];
              a[q] = x > y ? x : y;
            }
            Sel::sync();
            if (kp >= kNST) {
              for (int pr = 0; pr < npairs; ++pr)
                team_sort_desc<Sel>(slots + (2 * gap * pr) * kp, kp, kp, stt);
            } else {
              bitonic_network<Sel, uint64_t, true>(slots, kp, kp, npairs, 2 * gap * kp, stt);
            }
          }
        }
        if (stt == 0) TL_PIECE(j, 6);
        // the row's k-th word must lie above every speculative threshold its
        // pieces started from, else the row is selected again
        const uint64_t wk = slots[k - 1];
        Sel::sync();
        if (rs != 0ull && wk <= rs) {
          redo = true;
          redo_lb = wk;
        } else {
          write_row(p, pc.r, slots, stt, kNST);
        }
        Sel::sync();
        uint64_t* ib = par ? inbox1 : inbox0;
        for (int q = stt; q < kInbox; q += kNST) ib[q] = 0ull;  // empty slots again
        __threadfence_block();
        if (stt == 0) {
          p.row_theta[pc.r] = 0ull;
          p.row_spec[pc.r] = 0ull;
          atomicExch(&p.tickets[pc.r], 0u);
        }
      }
    }
    if (redo) {
      // (as a lone piece: the row's shared words are already reset)
      Piece lone = pc;
      lone.contributors = 1;
      if (stt == 0) TL_CNT(tlc, kCycSelRescan);
      rescan(lone, redo_lb);
      if (stt == 0) {
        atomicAdd(&p.sorts[pc.r], nsorts);
        atomicAdd(&p.survivors[pc.r], nsorted);
      }
      nsorts = 0;
      nsorted = 0;
      write_row(p, pc.r, kept, stt, kNST);
    }
    // a clean tray and threshold, then hand this parity back to the filters
    Sel::sync();
    for (int q = stt; q < kp; q += kNST) kept[q] = 0ull;
    tray_n = 0;
    kept_n = 0;
    pruned = 0;
    theta = 0ull;
    theta_proven = 0ull;
    Sel::sync();
    if (stt == 0) {
      *reinterpret_cast<volatile unsigned long long*>(&st.theta[par]) = 0ull;
      st.spec[par] = 0ull;
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&st.sel_pieces) = j + 1;
      TL_ACC(tlc, kCycSelEnd, cend);
      TL_PIECE(j, 3);
    }
  }
  timed_out = Sel::sync_or(timed_out);
  if (stt == 0 && timed_out) atomicOr(p.status, TOPK_STATUS_TIMEOUT);
  if (stt == 0) {
    TL_FLUSH(tlc);
    TL_SET(kTlSelExit, tl_now());
  }
#undef wl
}

__global__ void __launch_bounds__(32)
visit_order_kernel(int32_t m, int32_t row, int64_t first, uint32_t seed_lo, uint32_t seed_hi,
                   int32_t* out) {
  __shared__ uint32_t perm[kPermChunk];
  build_visit_order_warp(perm, m, first, row, seed_lo, seed_hi, false, threadIdx.x);
  for (int j = threadIdx.x; j < m; j += 32) out[j] = int32_t(perm[j] & uint32_t(kPermChunk - 1));
}

// ---------------------------------------------------------------------------
// Host side.

struct DeviceInfo {
  std::atomic<int> configured{0};
  int sms = 0;
};
DeviceInfo g_devices[64];

// The block pool's kernel (defined below) and its launch shape.
constexpr int kPoolSelThreads = 1024;
constexpr uint32_t kPoolSeg = 32 * kPoolSelThreads;  // blocks per output segment (one word a thread)
constexpr uint32_t kPoolCap = 8192;                  // keys the pool's fast path may collect
constexpr uint32_t kPoolWide = 4096;                  // bitmap words of the one-pass write (131,072 blocks)
constexpr int kPoolSmem =
    int(sizeof(uint32_t)) * (4096 + 2 * kPoolSelThreads + 2 * int(kPoolCap) + int(kPoolWide));
__global__ void __launch_bounds__(kPoolSelThreads) pool_select_kernel(
    const float* bmax, int64_t bstride, const int32_t* lengths, int64_t n, int32_t pool_blocks,
    int32_t pinned, int32_t* out_pool, uint32_t* status);

// The short-row kernel (defined below) and its launch shape.
constexpr int kShortThreads = 256;
constexpr int kShortPer = 16;                    // scores a thread tests per chunk
constexpr int kShortChunk = kShortThreads * kShortPer;  // elements a chunk (one bulk copy)
constexpr int kShortStages = 2;                  // chunk copies in flight per CTA
constexpr int kShortMaxN = 65536;                // longest row (valid length) of the path
constexpr int kShortCtasPerSm = 3;               // resident CTAs per SM at most
using Blk = Team<kShortThreads, 0>;              // (barrier 0 over the whole CTA)

// tray mark (words before a select) and capacity for kept-list size kp; the
// dynamic shared memory: tray, ring of chunk stages, their barriers
__host__ __device__ inline int short_mark(int kp) { return kp <= 512 ? 1024 : 2 * kp; }
__host__ __device__ inline int short_cap(int kp) { return short_mark(kp) + kShortChunk; }
__host__ __device__ inline int short_smem(int kp) {
  return short_cap(kp) * int(sizeof(uint64_t)) + kShortStages * kShortChunk * int(sizeof(float)) +
         kShortStages * int(sizeof(uint64_t));
}
__global__ void __launch_bounds__(kShortThreads, kShortCtasPerSm) short_select_kernel(const Params p);

cudaError_t configure_device(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  DeviceInfo* info = dev < 64 ? &g_devices[dev] : nullptr;
  if (info && info->configured.load()) {
    *sms = info->sms;
    return cudaSuccess;
  }
  int most = 0;
  for (int kp = 1; kp <= TOPK_MAX_K; kp <<= 1) most = max(most, smem_layout(kp).total);
  e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(pool_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kPoolSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(short_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           short_smem(TOPK_MAX_K));
  if (e != cudaSuccess) return e;
  int count = 0;
  e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  *sms = count;
  if (info) {
    info->sms = count;
    info->configured.store(1);
  }
  return cudaSuccess;
}

int32_t resolve_split(int32_t rows, int64_t n, int32_t split, int plan_sms) {
  return split == 0 ? auto_split(rows, n, plan_sms) : split;
}

// Partial-list slots a workspace is sized for: enough for any plan count up
// to kMaxFlatCtas (auto_split and the flat plan only grow with the count).
size_t sized_slots(int32_t rows, int64_t n, int32_t split) {
  return partial_slots(rows, split, resolve_split(rows, n, split, kMaxFlatCtas), kMaxFlatCtas);
}

// The planning count of the current device: its SM count, at most
// kMaxFlatCtas; kSmsDefault when no device can be queried.
int device_plan_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return kSmsDefault;
  }
  int v = cached[dev].load();
  if (v == 0) {
    int count = 0;
    if (cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        count < 1) {
      cudaGetLastError();
      return kSmsDefault;
    }
    v = count < kMaxFlatCtas ? count : kMaxFlatCtas;
    cached[dev].store(v);
  }
  return v;
}

// ---------------------------------------------------------------------------
// The layer-20 block pool around the selection (topk_select_pool).

constexpr int kPoolBlock = TOPK_POOL_BLOCK;  // positions per block

bool pool_args_ok(int32_t pool_blocks, int32_t pinned_blocks) {
  return pool_blocks >= 1 && pinned_blocks >= 0 && pinned_blocks <= pool_blocks &&
         pool_blocks - pinned_blocks <= TOPK_MAX_K;
}

// Workspace of topk_select_pool: the selection's own workspace first (its
// status word is the call's), then the block maxima (rows x bstride floats).
struct PoolLayout {
  int64_t nb, bstride;
  size_t bmax, total;
};

PoolLayout pool_layout(int32_t rows, int64_t n, int32_t k) {
  PoolLayout L;
  L.nb = (n + kPoolBlock - 1) / kPoolBlock;
  L.bstride = (L.nb + 3) & ~int64_t(3);  // 16-byte aligned rows
  L.bmax = align256(topk_ws_bytes_ex(rows, n, k, 0));
  L.total = align256(L.bmax + sizeof(float) * size_t(rows) * size_t(L.bstride));
  return L;
}

__device__ __forceinline__ int64_t pool_row_length(const int32_t* lengths, int32_t r, int64_t n) {
  if (!lengths) return n;
  const int64_t L = lengths[r];
  return L < 0 ? 0 : (L > n ? n : L);
}


// CTA-wide exclusive prefix sum of one value per thread (kPoolSelThreads
// threads); also returns the total.  Uses `scratch` (kPoolSelThreads / 32
// words) and ends with a barrier.
__device__ __forceinline__ uint32_t pool_scan(uint32_t v, uint32_t* scratch, uint32_t& total) {
  const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) scratch[wp] = incl;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int q = 0; q < kPoolSelThreads / 32; ++q) {
    const uint32_t c = scratch[q];
    before += q < wp ? c : 0u;
    all += c;
  }
  __syncthreads();
  total = all;
  return before + incl - v;
}


// One row's pool, one CTA per row: the best kb of the row's candidate blocks
// (its blocks that are not pinned), by the order key of each block maximum
// (key 0: the block has no score).  A radix select (12 + 12 + 8 bits) finds
// the exact key T of the kb-th block and how many blocks equal to T the pool
// takes (the first ones in index order); the blocks above T and those are
// written in ascending block order, then the pinned blocks, then -1.
//   Fast path: a sample (8 consecutive keys of every `stride`) gives a key
// that about 1.5 kb + 8 * stride / 8 of the row's keys reach; one pass over
// the row collects every key at or above it into shared memory, and the
// select and the ordered write run on that list.  If the list holds fewer
// than kb keys or overflows, the select and the write run over the whole row
// (three passes and a marking pass).
__global__ void __launch_bounds__(kPoolSelThreads) pool_select_kernel(
    const float* bmax, int64_t bstride, const int32_t* lengths, int64_t n, int32_t pool_blocks,
    int32_t pinned, int32_t* out_pool, uint32_t* status) {
  (void)status;
  extern __shared__ __align__(16) uint32_t psm[];
  uint32_t* hist = psm;                          // 4096 bins
  uint32_t* gtbits = psm + 4096;                 // output bitmaps, one word a thread
  uint32_t* eqbits = gtbits + kPoolSelThreads;
  uint32_t* lkey = eqbits + kPoolSelThreads;     // fast path: keys (the sample, then the list)
  uint32_t* lidx = lkey + kPoolCap;              // fast path: their block indices
  uint32_t* wide_eq = lidx + kPoolCap;           // one-pass write: blocks equal to T (with hist: above)
  __shared__ uint32_t scratch[kPoolSelThreads / 32];
  __shared__ uint32_t s_bin, s_above, s_n;
  const int32_t r = blockIdx.x;
  const int t = threadIdx.x, lane = t & 31;
  const int64_t nb = (pool_row_length(lengths, r, n) + kPoolBlock - 1) / kPoolBlock;
  const int32_t pe = int32_t(nb < pinned ? nb : pinned);
  const uint32_t nc = uint32_t(nb - pe);  // candidate blocks [0, nc)
  const uint32_t kb = uint32_t(pool_blocks - pe);
  const float* row = bmax + int64_t(r) * bstride;
  auto to_key = [](float v) -> uint32_t {
    const uint32_t bits = __float_as_uint(v);
    return (bits & 0x7FFFFFFFu) > 0x7F800000u ? 0u : order_key(bits);  // NaN: no score
  };
  // 16 keys a thread: four float4 loads in flight (row is 16-byte aligned)
  auto load16 = [&](uint32_t base, uint32_t (&key)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t b = base + 4u * kPoolSelThreads * uint32_t(q) + 4u * uint32_t(t);
      float4 v;
      if (b + 4u <= nc) {
        v = __ldg(reinterpret_cast<const float4*>(row + b));
      } else {
        const float nan = __int_as_float(0x7FC00000);
        v.x = b < nc ? row[b] : nan;
        v.y = b + 1u < nc ? row[b + 1u] : nan;
        v.z = b + 2u < nc ? row[b + 2u] : nan;
        v.w = b + 3u < nc ? row[b + 3u] : nan;
      }
      key[4 * q + 0] = to_key(v.x);
      key[4 * q + 1] = to_key(v.y);
      key[4 * q + 2] = to_key(v.z);
      key[4 * q + 3] = to_key(v.w);
    }
  };
  // histogram of keys in shared memory (key 0 = none)
  auto feed_smem = [&](const uint32_t* keys, uint32_t cnt, uint32_t prefix, uint32_t pmask, int sh,
                       uint32_t dmask) {
    for (uint32_t i = t; i < cnt; i += kPoolSelThreads) {
      const uint32_t k = keys[i];
      if (k != 0u && (k & pmask) == prefix) atomicAdd(&hist[(k >> sh) & dmask], 1u);
    }
  };
  auto block_of = [&](uint32_t base, int q) -> uint32_t {  // load16's key q
    return base + 4u * kPoolSelThreads * uint32_t(q >> 2) + 4u * uint32_t(t) + uint32_t(q & 3);
  };
  constexpr uint32_t kStep = 16u * kPoolSelThreads;

  // One radix select: `feed(prefix, pmask, sh, dmask)` adds the keys that
  // match the prefix into hist.  want >= 1.  Returns the key of the want-th
  // largest (0 and all = true when every key is taken) and in need how many
  // keys equal to it are taken.
  auto radix = [&](auto feed, uint32_t want, uint32_t& T, uint32_t& need, bool& all,
                   int passes = 3) {
    uint32_t prefix = 0, pmask = 0;
    need = want;
    all = false;
    for (int pass = 0; pass < passes; ++pass) {
      const int sh = pass == 0 ? 20 : (pass == 1 ? 8 : 0);  // digits of 12, 12 and 8 bits
      const uint32_t dmask = pass < 2 ? 0xFFFu : 0xFFu;
      for (int j = t; j < 4096; j += kPoolSelThreads) hist[j] = 0u;
      __syncthreads();
      feed(prefix, pmask, sh, dmask);
      __syncthreads();
      const int nbins = int(dmask) + 1;
      const int per = nbins >= kPoolSelThreads ? nbins / kPoolSelThreads : 1;
      const int top = nbins - 1 - t * per;
      uint32_t mine = 0;
      if (top >= 0)
        for (int q = 0; q < per; ++q) mine += hist[top - q];
      uint32_t total;
      const uint32_t above = pool_scan(mine, scratch, total);
      if (pass == 0 && total <= want) {
        all = true;
        break;
      }
      if (top >= 0 && above < need && above + mine >= need) {
        uint32_t acc = above;
        for (int q = 0; q < per; ++q) {
          const uint32_t c = hist[top - q];
          if (acc + c >= need) {
            s_bin = uint32_t(top - q);
            s_above = acc;
            break;
          }
          acc += c;
        }
      }
      __syncthreads();
      prefix |= s_bin << sh;
      pmask |= dmask << sh;
      need -= s_above;
      __syncthreads();
    }
    T = all ? 0u : prefix;
    if (all) need = 0u;
  };

  // Ascending output over segments of kPoolSeg blocks: `mark(s0, send)` sets
  // the bits of the blocks above T (gtbits) and equal to T (eqbits); a
  // selected block's place = blocks above T before it + min(blocks equal to
  // T before it, eq_take).  Returns how many blocks were written.
  int32_t* out = out_pool + int64_t(r) * pool_blocks;
  auto emit = [&](auto mark, uint32_t eq_take) -> uint32_t {
    uint32_t gt_run = 0, eq_run = 0;
    for (uint32_t s0 = 0; s0 < nc; s0 += kPoolSeg) {
      gtbits[t] = 0u;
      eqbits[t] = 0u;
      __syncthreads();
      mark(s0, min(nc, s0 + kPoolSeg));
      __syncthreads();
      const uint32_t g = gtbits[t], e = eqbits[t];
      uint32_t tot;
      const uint32_t before =
          pool_scan(uint32_t(__popc(g)) | (uint32_t(__popc(e)) << 16), scratch, tot);
      const uint32_t gb = gt_run + (before & 0xFFFFu), eb = eq_run + (before >> 16);
      uint32_t esel = 0u, left = eq_take > eb ? eq_take - eb : 0u;
      for (uint32_t m = e; m != 0u && left > 0u; m &= m - 1u, --left) esel |= m & (0u - m);
      uint32_t pos = gb + min(eb, eq_take);
      for (uint32_t m = g | esel; m != 0u; m &= m - 1u, ++pos)
        if (IN_BOUNDS(pos < uint32_t(pool_blocks), status))
          out[pos] = int32_t(s0 + 32u * uint32_t(t) + uint32_t(__ffs(m) - 1));
      gt_run += tot & 0xFFFFu;
      eq_run += tot >> 16;
      __syncthreads();
    }
    return gt_run + min(eq_run, eq_take);
  };
  auto set_bit = [&](uint32_t b, uint32_t s0, uint32_t key, uint32_t T) {
    const uint32_t w = (b - s0) >> 5, bit = 1u << ((b - s0) & 31u);
    if (key > T) atomicOr(&gtbits[w], bit);
    else if (key == T) atomicOr(&eqbits[w], bit);
  };

  uint32_t sel = 0;
  bool done = kb == 0 || nc == 0;
  if (!done) {
    // ---- fast path: sample, collect, select and write from the list ----
    uint32_t stride = 128;
    while (uint64_t(stride) * kPoolSelThreads < nc) stride <<= 1;  // one group a thread
    const uint32_t ngroups = (nc + stride - 1) / stride;
    if (ngroups * 8u <= kPoolCap) {
      // sample: keys [g * stride, g * stride + 8) of group g
      if (uint32_t(t) < ngroups) {
        const uint32_t b0 = uint32_t(t) * stride;  // a multiple of 128: 16-byte aligned
        if (b0 + 8u <= nc) {
          const float4 v0 = __ldg(reinterpret_cast<const float4*>(row + b0));
          const float4 v1 = __ldg(reinterpret_cast<const float4*>(row + b0 + 4u));
          lkey[8 * t + 0] = to_key(v0.x);
          lkey[8 * t + 1] = to_key(v0.y);
          lkey[8 * t + 2] = to_key(v0.z);
          lkey[8 * t + 3] = to_key(v0.w);
          lkey[8 * t + 4] = to_key(v1.x);
          lkey[8 * t + 5] = to_key(v1.y);
          lkey[8 * t + 6] = to_key(v1.z);
          lkey[8 * t + 7] = to_key(v1.w);
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t b = b0 + uint32_t(c);
            lkey[8 * t + c] = b < nc ? to_key(row[b]) : 0u;
          }
        }
      }
      __syncthreads();
      const uint32_t scount = ngroups * 8u;
      // the sample key that about 1.5 kb + stride of the row's keys reach
      const uint64_t want64 = (3ull * kb * 8ull + 2ull * stride - 1ull) / (2ull * stride) + 8ull;
      uint32_t T0 = 0, e0 = 0;
      bool all0 = false;
      if (want64 <= scount) {
        // (two passes: a 24-bit prefix is bound enough -- its bin's lower
        // edge only lets a few more keys into the list)
        radix([&](uint32_t prefix, uint32_t pmask, int sh, uint32_t dmask) {
                feed_smem(lkey, scount, prefix, pmask, sh, dmask);
              }, uint32_t(want64), T0, e0, all0, 2);
      }
      // collect every key >= T0 (all keys when the sample cannot bound them)
      if (t == 0) s_n = 0u;
      __syncthreads();
      const uint32_t lo = all0 || want64 > scount ? 1u : max(T0, 1u);  // (0: no score)
      for (uint32_t base = 0; base < nc; base += kStep) {
        uint32_t key[16];
        load16(base, key);
        uint32_t c = 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) c += (key[q] >= lo && block_of(base, q) < nc) ? 1u : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
          if (lane >= d) incl += o;
        }
        uint32_t wbase = 0;
        if (lane == 31 && incl) wbase = atomicAdd(&s_n, incl);
        wbase = __shfl_sync(0xFFFFFFFFu, wbase, 31);
        uint32_t at = wbase + incl - c;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const uint32_t b = block_of(base, q);
          if (key[q] >= lo && b < nc) {
            if (at < kPoolCap) {
              lkey[at] = key[q];
              lidx[at] = b;
            }
            ++at;
          }
        }
      }
      __syncthreads();
      const uint32_t nl = s_n;
      if (nl >= kb && nl <= kPoolCap) {
        uint32_t T, eq_take;
        bool all;
        radix([&](uint32_t prefix, uint32_t pmask, int sh, uint32_t dmask) {
                feed_smem(lkey, nl, prefix, pmask, sh, dmask);
              }, kb, T, eq_take, all);
        if (nc <= 32u * kPoolWide) {
          // one pass: bitmaps of the whole row (hist: blocks above T, wide_eq:
          // blocks equal to T), four words a thread, one packed prefix scan
          uint32_t* gtw = hist;
          for (uint32_t j = t; j < kPoolWide; j += kPoolSelThreads) {
            gtw[j] = 0u;
            wide_eq[j] = 0u;
          }
          __syncthreads();
          for (uint32_t i = t; i < nl; i += kPoolSelThreads) {
            const uint32_t b = lidx[i], key = lkey[i], bit = 1u << (b & 31u);
            if (key > T) atomicOr(&gtw[b >> 5], bit);
            else if (key == T) atomicOr(&wide_eq[b >> 5], bit);
          }
          __syncthreads();
          constexpr int kW = int(kPoolWide) / kPoolSelThreads;  // words a thread
          uint32_t gs = 0, es = 0;
#pragma unroll
          for (int q = 0; q < kW; ++q) {
            gs += uint32_t(__popc(gtw[kW * t + q]));
            es += uint32_t(__popc(wide_eq[kW * t + q]));
          }
          uint32_t tot;
          const uint32_t before = pool_scan(gs | (es << 16), scratch, tot);
          uint32_t gb = before & 0xFFFFu, eb = before >> 16;
#pragma unroll
          for (int q = 0; q < kW; ++q) {
            const uint32_t w = uint32_t(kW * t + q);
            const uint32_t g = gtw[w], e = wide_eq[w];
            uint32_t esel = 0u, left = eq_take > eb ? eq_take - eb : 0u;
            for (uint32_t m = e; m != 0u && left > 0u; m &= m - 1u, --left) esel |= m & (0u - m);
            uint32_t pos = gb + min(eb, eq_take);
            for (uint32_t m = g | esel; m != 0u; m &= m - 1u, ++pos)
              if (IN_BOUNDS(pos < uint32_t(pool_blocks), status))
                out[pos] = int32_t(32u * w + uint32_t(__ffs(m) - 1));
            gb += uint32_t(__popc(g));
            eb += uint32_t(__popc(e));
          }
          sel = (tot & 0xFFFFu) + min(tot >> 16, eq_take);
        } else {
          sel = emit([&](uint32_t s0, uint32_t send) {
                       for (uint32_t i = t; i < nl; i += kPoolSelThreads) {
                         const uint32_t b = lidx[i];
                         if (b >= s0 && b < send) set_bit(b, s0, lkey[i], T);
                       }
                     }, eq_take);
        }
        done = true;
      }
    }
  }
  if (!done) {
    // ---- whole-row path ----
    uint32_t T, eq_take;
    bool all;
    radix([&](uint32_t prefix, uint32_t pmask, int sh, uint32_t dmask) {
            for (uint32_t base = 0; base < nc; base += kStep) {
              uint32_t key[16];
              load16(base, key);
              bool any = false;
#pragma unroll
              for (int q = 0; q < 16; ++q) any |= key[q] != 0u && (key[q] & pmask) == prefix;
              if (!__any_sync(0xFFFFFFFFu, any)) continue;
#pragma unroll
              for (int q = 0; q < 16; ++q)
                if (key[q] != 0u && (key[q] & pmask) == prefix)
                  atomicAdd(&hist[(key[q] >> sh) & dmask], 1u);
            }
          }, kb, T, eq_take, all);
    sel = emit([&](uint32_t s0, uint32_t send) {
                 for (uint32_t base = s0; base < send; base += kStep) {
                   uint32_t key[16];
                   load16(base, key);
#pragma unroll
                   for (int q = 0; q < 16; ++q) {
                     const uint32_t b = block_of(base, q);
                     if (b < send && key[q] != 0u) set_bit(b, s0, key[q], T);
                   }
                 }
               }, eq_take);
  }
  for (int j = t; j < pool_blocks; j += kPoolSelThreads) {
    if (uint32_t(j) < sel) continue;
    out[j] = uint32_t(j) < sel + uint32_t(pe) ? int32_t(nb - pe) + (j - int32_t(sel)) : -1;
  }
}

// The queue plan's order: rows sorted by unit count, longest first (a
// counting sort; rows of equal length in any order -- results never depend
// on the order).  One CTA; unit counts up to kQueueMaxUnits.
__global__ void __launch_bounds__(kPoolSelThreads) queue_order_kernel(
    const int32_t* lengths, int32_t rows, int64_t n, int32_t u_full, int32_t* order) {
  __shared__ uint32_t cnt[kQueueMaxUnits + 1];
  __shared__ uint32_t scratch[kPoolSelThreads / 32];
  const int t = threadIdx.x;
  for (int j = t; j <= u_full; j += kPoolSelThreads) cnt[j] = 0u;
  __syncthreads();
  auto bin = [&](int32_t r) -> int {  // longest first: bin 0 holds the longest rows
    const int64_t L = pool_row_length(lengths, r, n);
    return u_full - int((L + kUnit - 1) / kUnit);
  };
  for (int32_t r = t; r < rows; r += kPoolSelThreads) atomicAdd(&cnt[bin(r)], 1u);
  __syncthreads();
  constexpr int kPer = (kQueueMaxUnits + 1 + kPoolSelThreads - 1) / kPoolSelThreads;
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int j = t * kPer + q;
    c[q] = j <= u_full ? cnt[j] : 0u;
    sum += c[q];
  }
  uint32_t total;
  uint32_t off = pool_scan(sum, scratch, total);  // (ends with a barrier)
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int j = t * kPer + q;
    if (j <= u_full) cnt[j] = off;
    off += c[q];
  }
  __syncthreads();
  for (int32_t r = t; r < rows; r += kPoolSelThreads) order[atomicAdd(&cnt[bin(r)], 1u)] = r;
}

// ---------------------------------------------------------------------------
// Short rows (batches of many rows of at most kShortMaxN elements, the
// prefill's causal rows): the same method -- a threshold that only rises, a
// tray of the words above it, a select that raises it when the tray passes
// its mark, a bitonic sort of the survivors at the end -- run by one 256-
// thread CTA per row with no role split, several CTAs per SM, rows taken
// from the shared queue (longest first).  A row of a few units would spend
// most of the selection kernel's per-piece work (warm start, two-inbox
// hand-over, piece end) waiting for its selector team; here thread 0 copies
// the row in 4096-element chunks (one cp.async.bulk each) into a two-stage
// ring, every thread tests its sixteen scores of a chunk, and the row's first
// chunk, met with an empty threshold, sets the first one through the select.
// Rows are not visited in a shuffled order: a row is at most sixteen chunks.

struct ShortState {
  uint32_t hist[256];
  int cnt;        // tray words (append counter)
  int row;        // the queue item this CTA works on
  int sel_b, sel_above, sel_binc;
};

// The exact best-k prefix of the tray's n words (all distinct, n > k): a
// byte-wise radix select from the top byte finds a prefix T such that exactly
// k words are >= T; those k words are compacted to the tray's front (a word
// only moves down, and each round reads all its words before any is written).
// Returns T.  Ends with a barrier.
__device__ uint64_t short_select(uint64_t* tray, int n, int k, ShortState& st, int t,
                                 uint32_t* status) {
  const int lane = t & 31, warp = t >> 5;
  uint64_t prefix = 0ull;
  uint32_t need = uint32_t(k);
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    const uint64_t hmask = pass == 0 ? 0ull : (~0ull << (shift + 8));
    for (int b = t; b < 256; b += kShortThreads) st.hist[b] = 0u;
    Blk::sync();
    for (int j = t; j < n; j += kShortThreads) {
      const uint64_t w = tray[j];
      if ((w & hmask) == prefix) atomicAdd(&st.hist[uint32_t(w >> shift) & 0xFFu], 1u);
    }
    Blk::sync();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l, scanned from the top
      uint32_t c8[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c8[q] = st.hist[255 - 8 * lane - q];
        sum += c8[q];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
      }
      const uint32_t excl = incl - sum;
      if (excl < need && incl >= need) {
        uint32_t acc = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (acc < need && acc + c8[q] >= need) {
            st.sel_b = 255 - 8 * lane - q;
            st.sel_above = int(acc);
            st.sel_binc = int(c8[q]);
          }
          acc += c8[q];
        }
      }
    }
    Blk::sync();
    const uint32_t b = uint32_t(st.sel_b), above = uint32_t(st.sel_above),
                   binc = uint32_t(st.sel_binc);
    prefix |= uint64_t(b) << shift;
    need -= above;
    if (binc == need) break;  // the whole bin is in: exactly k words are >= prefix
  }
  const uint64_t T = prefix;
  if (t == 0) st.cnt = 0;
  Blk::sync();
  constexpr int R = 8;
  for (int base0 = 0; base0 < n; base0 += R * kShortThreads) {
    uint64_t w[R];
    bool keep[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int j = base0 + u * kShortThreads + t;
      w[u] = j < n ? tray[j] : 0ull;
      keep[u] = j < n && w[u] >= T;
    }
    Blk::sync();
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, keep[u]);
      if (mask) {
        int at = 0;
        if (lane == 0) at = atomicAdd(&st.cnt, __popc(mask));
        at = __shfl_sync(0xFFFFFFFFu, at, 0);
        const int pos = at + __popc(mask & ((1u << lane) - 1u));
        if (keep[u] && IN_BOUNDS(pos < n, status)) tray[pos] = w[u];
      }
    }
  }
  Blk::sync();
  return T;
}

__global__ void __launch_bounds__(kShortThreads, kShortCtasPerSm) short_select_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem_s[];
  const int k = p.k, kp = p.kp;
  const int mark = short_mark(kp), cap = short_cap(kp);
  uint64_t* tray = reinterpret_cast<uint64_t*>(smem_s);
  float* ring = reinterpret_cast<float*>(smem_s + size_t(cap) * sizeof(uint64_t));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kShortStages * kShortChunk);
  __shared__ ShortState st;
  const int t = threadIdx.x, lane = t & 31;
  if (t == 0) {
    grid_dep_launch();
    for (int q = 0; q < kShortStages; ++q) mbar_init(&full[q], 1);
    mbar_init_fence();
  }
  Blk::sync();
  grid_dep_wait();  // (global memory only after the stream's previous grid)
  const uint32_t total = uint32_t(p.rows);
  const uint64_t l2pol = l2_policy_evict_first();
  bool saw_nan = false, timed_out = false;
  uint32_t g_issue = 0, g_use = 0;  // chunks issued (thread 0) and consumed, over the CTA's rows
#if TOPK_TIMELINE
  // (thread 0's cycle sums, see TlShort)
  unsigned long long tls[kTlShortEndSlot - kTlShortRows] = {};
  const long long tl_c0 = clock64();
  long long tl_a = tl_c0;
#define TLS_MARK(slot)                                      \
  do {                                                      \
    const long long tl_b = clock64();                       \
    tls[(slot) - kTlShortRows] += (unsigned long long)(tl_b - tl_a); \
    tl_a = tl_b;                                            \
  } while (0)
#define TLS_COUNT(slot, v) (tls[(slot) - kTlShortRows] += (unsigned long long)(v))
#else
#define TLS_MARK(slot) ((void)0)
#define TLS_COUNT(slot, v) ((void)0)
#endif
  for (;;) {
    if (t < 32) {
      const uint32_t q = queue_take(p.queue, total);
      if (t == 0) st.row = int(q);
    }
    if (t == 0) st.cnt = 0;
    Blk::sync();
    const uint32_t item = uint32_t(st.row);
    if (item >= total) break;
    const int32_t r = p.order ? p.order[item] : int32_t(item);
    int64_t L = p.lengths ? int64_t(p.lengths[r]) : p.n;
    if (L < 0 || L > p.n) {
      if (t == 0) atomicOr(p.status, TOPK_STATUS_BAD_LENGTH);
      L = L < 0 ? 0 : p.n;
    }
    const uint32_t Lu = uint32_t(L);
    const uint32_t nc = (Lu + uint32_t(kShortChunk) - 1) / uint32_t(kShortChunk);
    const float* row = p.scores + int64_t(r) * p.row_stride;
    const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    // elements of chunk c in its stage (a 16-byte multiple; the rest, past
    // it, come from global memory)
    auto copied_of = [&](uint32_t c) -> uint32_t {
      const uint32_t left = Lu - c * uint32_t(kShortChunk);
      return aligned ? (min(left, uint32_t(kShortChunk)) & ~3u) : 0u;
    };
    // thread 0: chunk c of this row into the next stage
    auto issue = [&](uint32_t c) {
      const int stage = int(g_issue % uint32_t(kShortStages));
      const uint32_t bytes = copied_of(c) * 4u;
      fence_proxy_async_smem();
      if (bytes) {
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_load_hint(ring + stage * kShortChunk, row + size_t(c) * kShortChunk, bytes,
                       &full[stage], l2pol);
      } else {
        mbar_arrive(&full[stage]);
      }
      ++g_issue;
    };
    uint64_t theta = 0ull;  // words above it are admitted (0: every real word)
    int tray_n = 0;
    uint32_t admitted = 0;
    TLS_MARK(kTlShortMeta);
    TLS_COUNT(kTlShortRows, 1);
    {
      if (t == 0)
        for (uint32_t c = 0; c < nc && c < uint32_t(kShortStages); ++c) issue(c);
      for (uint32_t c = 0; c < nc; ++c) {
        TLS_COUNT(kTlShortNChunks, 1);
        const uint32_t c0 = c * uint32_t(kShortChunk);
        const int stage = int(g_use % uint32_t(kShortStages));
#if TOPK_TIMELINE
        const long long tl_w = clock64();
#endif
        if (!mbar_wait(&full[stage], (g_use / uint32_t(kShortStages)) & 1u,
                       timed_out ? 1u : kWaitLimit))
          timed_out = true;
        TLS_COUNT(kTlShortWait, clock64() - tl_w);
        ++g_use;
        const uint32_t copied = copied_of(c);
        const float* src = ring + stage * kShortChunk;
        // kShortPer scores a thread: float4 u of the chunk is t + kShortThreads u
        float x[kShortPer];
#pragma unroll
        for (int u = 0; u < kShortPer / 4; ++u) {
          const uint32_t q4 = uint32_t(4 * (t + kShortThreads * u));
          if (q4 + 4u <= copied) {
            const float4 v = reinterpret_cast<const float4*>(src)[t + kShortThreads * u];
            x[4 * u + 0] = v.x;
            x[4 * u + 1] = v.y;
            x[4 * u + 2] = v.z;
            x[4 * u + 3] = v.w;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t q = q4 + uint32_t(j);
              x[4 * u + j] = q < copied ? src[q]
                             : c0 + q < Lu ? __ldcs(row + c0 + q)
                                           : __int_as_float(0x7FFFFFFF);  // past the end: a NaN
            }
          }
        }
#pragma unroll
        for (int e = 0; e < kShortPer; ++e) {
          const uint32_t pos = c0 + uint32_t(4 * (t + kShortThreads * (e >> 2)) + (e & 3));
          const uint32_t bits = __float_as_uint(x[e]);
          const bool nan = (bits & 0x7FFFFFFFu) > 0x7F800000u;
          saw_nan |= nan && pos < Lu;
          const uint64_t w = (uint64_t(order_key(bits)) << 32) | uint64_t(~pos);
          const bool keep = !nan && w > theta;
          const uint32_t mask = __ballot_sync(0xFFFFFFFFu, keep);
          if (mask) {
            int at = 0;
            if (lane == 0) at = atomicAdd(&st.cnt, __popc(mask));
            at = __shfl_sync(0xFFFFFFFFu, at, 0);
            const int j = at + __popc(mask & ((1u << lane) - 1u));
            if (keep && IN_BOUNDS(j < cap, p.status)) tray[j] = w;
          }
        }
        Blk::sync();  // (the stage is read: it may take the row's next chunk)
        if (t == 0 && c + uint32_t(kShortStages) < nc) issue(c + uint32_t(kShortStages));
        admitted += uint32_t(st.cnt - tray_n);  // the words this chunk sent to the tray
        tray_n = st.cnt;
        // Every thread reads the count before any thread's next appends change
        // it (the select begins with a barrier of its own): a warp that read it
        // late would see the next chunk's words and leave the others' barriers.
        if (tray_n > mark) {
          TLS_MARK(kTlShortChunks);
          TLS_COUNT(kTlShortNSelects, 1);
          // keep the best k of everything seen so far; the threshold rises
          const uint64_t T = short_select(tray, tray_n, k, st, t, p.status);
          theta = T - 1ull;
          tray_n = k;
          TLS_MARK(kTlShortSelect);
        } else {
          Blk::sync();
        }
      }
    }
    TLS_MARK(kTlShortChunks);
    // the exact best k, sorted, to the row (empty words past the survivors)
    if (tray_n > k) {
      short_select(tray, tray_n, k, st, t, p.status);
      tray_n = k;
    }
    const int P = max(next_pow2_dev(max(tray_n, 1)), kShortThreads);
    for (int j = tray_n + t; j < max(P, k); j += kShortThreads) tray[j] = 0ull;
    Blk::sync();
    team_sort_desc<Blk>(tray, P, 2, t);
    write_row(p, r, tray, t, kShortThreads);
    if (t == 0) {
      atomicAdd(&p.sorts[r], 1u);
      atomicAdd(&p.survivors[r], uint32_t(tray_n));
      atomicAdd(&p.admitted[r], admitted);
    }
    Blk::sync();  // (the tray and the queue word are rewritten for the next row)
    TLS_MARK(kTlShortEnd);
  }
  if (__any_sync(0xFFFFFFFFu, saw_nan) && lane == 0) atomicOr(p.status, TOPK_STATUS_NAN);
  if (__any_sync(0xFFFFFFFFu, timed_out) && lane == 0) atomicOr(p.status, TOPK_STATUS_TIMEOUT);
#if TOPK_TIMELINE
  if (t == 0) {
    tls[kTlShortTotal - kTlShortRows] = (unsigned long long)(clock64() - tl_c0);
    for (int q = 0; q < kTlShortEndSlot - kTlShortRows; ++q) TL_SET(kTlShortRows + q, tls[q]);
  }
#endif
#undef TLS_MARK
#undef TLS_COUNT
}

}  // namespace
}  // namespace topk

using namespace topk;

// ---------------------------------------------------------------------------
// Workspace for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they select:
// real-time paths that forbid allocation once running (an allocation can
// block on the driver), and plug-ins whose host framework owns every
// allocation and hands out only input and output buffers.  For them
// topk_select_noalloc uses this file-scope device array as its workspace.
// Every GPU that loads this library keeps the array (kNoAllocWsBytes) until
// the process exits.  In host code `g_noalloc_ws` names a host-side stand-in,
// not device memory: its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current.
constexpr size_t kNoAllocWsBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocWsBytes];

namespace {

struct NoAllocSlot {
  std::atomic<int> ready{0};
  void* ptr = nullptr;
};
NoAllocSlot g_noalloc_slots[64];

// Device address of the static workspace on the current device (set up on
// the first call per device, with that device current).
cudaError_t noalloc_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  NoAllocSlot& slot = g_noalloc_slots[dev];
  if (!slot.ready.load()) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_ws);
    if (e != cudaSuccess) return e;
    slot.ptr = ptr;
    slot.ready.store(1);
  }
  *out = slot.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" {

int topk_select_noalloc(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                        const int32_t* lengths_or_null, int32_t k, float* out_vals,
                        int32_t* out_idx, uint32_t* status_or_null, void* stream) {
  if (!shape_ok(rows, n, k) || row_stride < n) return TOPK_ERR_SHAPE;
  if (rows == 0) return TOPK_OK;
  const size_t need = topk_ws_bytes_ex(rows, n, k, 0);
  if (need == 0) return TOPK_ERR_SHAPE;
  if (need > kNoAllocWsBytes) return TOPK_ERR_NOSPACE;
  void* ws = nullptr;
  if (noalloc_ws_address(&ws) != cudaSuccess) return TOPK_ERR_LAUNCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word, tickets,
  // counters and row thresholds (everything before the partial lists) must
  // start at zero.
  const WsLayout wl = ws_layout(rows, next_pow2(k), sized_slots(rows, n, 0));
  if (cudaMemsetAsync(ws, 0, wl.partials, st) != cudaSuccess) return TOPK_ERR_LAUNCH;
  const int rc = topk_select(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx,
                             ws, stream);
  if (rc != TOPK_OK) return rc;
  if (status_or_null &&
      cudaMemcpyAsync(status_or_null, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
    return TOPK_ERR_LAUNCH;
  return TOPK_OK;
}

}  // extern "C"

extern "C" {

int32_t topk_split_plan(int32_t rows, int64_t n) {
  if (!shape_ok(rows, n, 1)) return 0;
  return auto_split(rows, n, device_plan_sms());
}

size_t topk_ws_bytes_ex(int32_t rows, int64_t n, int32_t k, int32_t split) {
  if (!shape_ok(rows, n, k) || split < 0 || split > kMaxSplit) return 0;
  return ws_layout(rows, next_pow2(k), sized_slots(rows, n, split)).total;
}

size_t topk_ws_bytes(int32_t rows, int64_t n, int32_t k) {
  return topk_ws_bytes_ex(rows, n, k, 0);
}

// The selection launch; `bmax` (block pool maxima, null for none) serves
// topk_select_pool.
static int launch_select(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                         const int32_t* lengths_or_null, int32_t k, float* out_vals,
                         int32_t* out_idx, void* ws, void* stream, int32_t split, uint64_t seed,
                         uint32_t flags, float* bmax, int64_t bstride) {
  if (!shape_ok(rows, n, k) || row_stride < n || split < 0 || split > kMaxSplit)
    return TOPK_ERR_SHAPE;
  if (rows == 0) return TOPK_OK;
  if (!scores || !out_vals || !out_idx) return TOPK_ERR_NULL;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return TOPK_ERR_WS;

  int sms = kSmsDefault;
  if (configure_device(&sms) != cudaSuccess) return TOPK_ERR_LAUNCH;
  const int plan_sms = sms < kMaxFlatCtas ? sms : kMaxFlatCtas;
  const int32_t S = resolve_split(rows, n, split, plan_sms);
  const int32_t kp = next_pow2(k);
  // (the partial lists come last: the other offsets do not depend on the
  // slot count, which is at most the sized one)
  const WsLayout wl = ws_layout(rows, kp, sized_slots(rows, n, split));
  const int64_t u_full = (n + kUnit - 1) / kUnit;

  unsigned char* w = static_cast<unsigned char*>(ws);
  Params p;
  p.scores = scores;
  p.row_stride = row_stride;
  p.n = n;
  p.lengths = lengths_or_null;
  p.rows = rows;
  p.k = k;
  p.kp = kp;
  p.nstage = ring_stages(kp);
  p.split = S;
  p.seg_units = int32_t((u_full + S - 1) / S);
  p.u_full = int32_t(u_full);
  p.out_vals = out_vals;
  p.out_idx = out_idx;
  p.status = reinterpret_cast<uint32_t*>(w);
  p.bmax = bmax;
  p.bstride = bstride;
  p.tickets = reinterpret_cast<uint32_t*>(w + wl.tickets);
  p.survivors = reinterpret_cast<uint32_t*>(w + wl.survivors);
  p.sorts = reinterpret_cast<uint32_t*>(w + wl.sorts);
  p.admitted = reinterpret_cast<uint32_t*>(w + wl.admitted);
  p.row_theta = reinterpret_cast<unsigned long long*>(w + wl.theta);
  p.row_spec = reinterpret_cast<unsigned long long*>(w + wl.spec);
  p.partials = reinterpret_cast<uint64_t*>(w + wl.partials);
  p.nslots = int64_t(partial_slots(rows, split, S, plan_sms));
  p.seed_lo = uint32_t(seed);
  p.seed_hi = uint32_t(seed >> 32);
  p.flags = flags;
  const bool stall = (flags & TOPK_FLAG_TEST_STALL) != 0;
  p.wait_limit = stall ? kTestWaitLimit : kWaitLimit;
  p.stall_at = stall ? kTestStallStage : -1;

  const int64_t cap = plan_sms;
  int64_t G;
  const bool flat = split == 0 && lengths_or_null == nullptr && rows < plan_sms;
  if (flat) {
    // one CTA per SM, equal shares of the batch's units: at least one CTA
    // per row, and rows split only into shares of kMinFlatUnits or more
    // (a split row ends in a leader merge of its CTAs' lists)
    const int64_t M = int64_t(rows) * u_full;
    G = cap;
    int64_t by_len = (M + kMinFlatUnits - 1) / kMinFlatUnits;
    if (by_len < rows) by_len = rows;
    if (G > by_len) G = by_len;
    p.plan = kPlanFlat;
    p.split = 1;
  } else {
    // (row, segment) items for one CTA per SM: dealt round-robin, or, for
    // batches of many rows, taken from a shared queue with the longest rows
    // first (a CTA that drew short rows takes more of them)
    const int64_t items = int64_t(rows) * S;
    G = items < cap ? items : cap;
    p.plan = rows >= plan_sms ? kPlanQueue : kPlanItems;
  }
  if (G < 1) G = 1;
  p.queue = reinterpret_cast<uint32_t*>(w + wl.queue);
  p.order = nullptr;
  if (p.plan == kPlanQueue && lengths_or_null && u_full <= kQueueMaxUnits) {
    int32_t* order = reinterpret_cast<int32_t*>(w + wl.order);
    queue_order_kernel<<<1, kPoolSelThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        lengths_or_null, rows, n, int32_t(u_full), order);
    if (cudaGetLastError() != cudaSuccess) return TOPK_ERR_LAUNCH;
    p.order = order;
  }
  // Many short rows (the queue plan, rows of at most kShortMaxN elements, no
  // block pool): one CTA per row, several CTAs per SM.
  const bool short_rows = p.plan == kPlanQueue && n <= kShortMaxN && bmax == nullptr &&
                          (flags & TOPK_FLAG_TEST_STALL) == 0;
  // Launched with programmatic stream serialization: the grid may start while
  // the stream's previous grid finishes (its set-up and, for the flat plan, its
  // plan and first visiting keys overlap that grid's tail); it reads global
  // memory only after that grid has completed (griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(G));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem_layout(kp).total);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (short_rows) {
    // resident CTAs per SM as the shared memory allows (227 KB, 1 KB each reserved)
    const int per_sm = min(kShortCtasPerSm, (227 * 1024) / (short_smem(kp) + 1024 + int(sizeof(ShortState))));
    const int64_t ctas = int64_t(sms) * (per_sm > 0 ? per_sm : 1);
    cfg.gridDim = dim3(unsigned(rows < ctas ? rows : ctas));
    cfg.blockDim = dim3(kShortThreads);
    cfg.dynamicSmemBytes = size_t(short_smem(kp));
    if (cudaLaunchKernelEx(&cfg, short_select_kernel, p) != cudaSuccess) return TOPK_ERR_LAUNCH;
    return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_LAUNCH;
  }
  if (cudaLaunchKernelEx(&cfg, topk_select_kernel, p) != cudaSuccess) return TOPK_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_LAUNCH;
}

int topk_select_ex(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                   const int32_t* lengths_or_null, int32_t k, float* out_vals, int32_t* out_idx,
                   void* ws, void* stream, int32_t split, uint64_t seed, uint32_t flags) {
  return launch_select(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx, ws,
                       stream, split, seed, flags, nullptr, 0);
}

int topk_select(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                const int32_t* lengths_or_null, int32_t k, float* out_vals, int32_t* out_idx,
                void* ws, void* stream) {
  return topk_select_ex(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx, ws,
                        stream, 0, kDefaultSeed, 0u);
}

size_t topk_pool_ws_bytes(int32_t rows, int64_t n, int32_t k, int32_t pool_blocks,
                          int32_t pinned_blocks) {
  if (!shape_ok(rows, n, k) || !pool_args_ok(pool_blocks, pinned_blocks)) return 0;
  return pool_layout(rows, n, k).total;
}

int topk_select_pool(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                     const int32_t* lengths_or_null, int32_t k, float* out_vals,
                     int32_t* out_idx, int32_t pool_blocks, int32_t pinned_blocks,
                     int32_t* out_pool, void* ws, void* stream) {
  if (!shape_ok(rows, n, k) || row_stride < n) return TOPK_ERR_SHAPE;
  if (!pool_args_ok(pool_blocks, pinned_blocks)) return TOPK_ERR_ARG;
  if (rows == 0) return TOPK_OK;
  if (!scores || !out_vals || !out_idx || !out_pool) return TOPK_ERR_NULL;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return TOPK_ERR_WS;
  const PoolLayout pl = pool_layout(rows, n, k);
  unsigned char* w = static_cast<unsigned char*>(ws);
  float* bmax = reinterpret_cast<float*>(w + pl.bmax);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one pass over the scores: the top-k and every block's maximum
  int rc = launch_select(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx, w,
                         stream, 0, kDefaultSeed, 0u, bmax, pl.bstride);
  if (rc != TOPK_OK) return rc;
  // the best blocks among each row's blocks that are not pinned, and the pool
  pool_select_kernel<<<rows, kPoolSelThreads, kPoolSmem, st>>>(
      bmax, pl.bstride, lengths_or_null, n, pool_blocks, pinned_blocks, out_pool,
      reinterpret_cast<uint32_t*>(w));
  return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_LAUNCH;
}

int topk_ws_status(void* ws, uint32_t* status_out, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return TOPK_ERR_WS;
  if (!status_out) return TOPK_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return TOPK_ERR_LAUNCH;
  if (cudaMemcpy(status_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TOPK_ERR_LAUNCH;
  if (cudaMemset(ws, 0, sizeof(uint32_t)) != cudaSuccess) return TOPK_ERR_LAUNCH;
  return TOPK_OK;
}

int topk_ws_stats(void* ws, int32_t rows, int64_t n, int32_t k, int32_t split,
                  uint32_t* survivors_out, uint32_t* sorts_out, uint32_t* admitted_out,
                  void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return TOPK_ERR_WS;
  if (!shape_ok(rows, n, k) || split < 0 || split > kMaxSplit) return TOPK_ERR_SHAPE;
  const WsLayout wl = ws_layout(rows, next_pow2(k), sized_slots(rows, n, split));
  unsigned char* w = static_cast<unsigned char*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return TOPK_ERR_LAUNCH;
  const size_t bytes = sizeof(uint32_t) * size_t(rows);
  uint32_t* outs[3] = {survivors_out, sorts_out, admitted_out};
  const size_t offs[3] = {wl.survivors, wl.sorts, wl.admitted};
  for (int i = 0; i < 3; ++i) {
    if (outs[i] &&
        cudaMemcpy(outs[i], w + offs[i], bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
      return TOPK_ERR_LAUNCH;
    if (cudaMemset(w + offs[i], 0, bytes) != cudaSuccess) return TOPK_ERR_LAUNCH;
  }
  return TOPK_OK;
}

int topk_timeline_read(unsigned long long* host_out, void* stream) {
#if TOPK_TIMELINE
  static_assert(kTlCtas == TOPK_TIMELINE_CTAS && kTlSlots == TOPK_TIMELINE_SLOTS,
                "timeline table shape");
  if (!host_out) return TOPK_ERR_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TOPK_ERR_LAUNCH;
  void* dev = nullptr;
  if (cudaGetSymbolAddress(&dev, g_timeline) != cudaSuccess) return TOPK_ERR_LAUNCH;
  const size_t bytes = sizeof(unsigned long long) * size_t(kTlCtas) * size_t(kTlSlots);
  if (cudaMemcpy(host_out, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
    return TOPK_ERR_LAUNCH;
  if (cudaMemset(dev, 0, bytes) != cudaSuccess) return TOPK_ERR_LAUNCH;
  return TOPK_OK;
#else
  (void)host_out;
  (void)stream;
  return TOPK_ERR_ARG;
#endif
}

int topk_visit_order(int32_t m, int32_t row, int64_t first_unit, uint64_t seed,
                     int32_t* order_out, void* stream) {
  if (m < 1 || m > kPermChunk || !order_out || first_unit < 0) return TOPK_ERR_ARG;
  visit_order_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      m, row, first_unit, uint32_t(seed), uint32_t(seed >> 32), order_out);
  return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_LAUNCH;
}

}  // extern "C"
