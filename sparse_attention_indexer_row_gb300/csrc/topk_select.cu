// Batched row-wise top-k for a sparse-attention indexer, GB300 (sm_103a).
//
// The selector streams every score of a row exactly once, in 1024-element
// blocks visited in a seeded shuffled order, and asks each element one
// question: does it beat the row's threshold?  Survivors go to a small
// shared-memory tray; when the tray passes its high-water mark a bitonic sort
// runs on the tray only, keeps the best k and raises the threshold to the k-th
// of them; the threshold never falls.  (The Secret GPU Kernel Behind DeepSeek
// V4.1 Flash, video transcript 3:18-4:20; the shuffle 3:30 and 4:55-5:10; the
// 32-bit survivor mask 5:10-5:22; the split-row leader merge 5:33-5:45.)
//
// GB300 mapping:
//  * Work is cut into pieces (a run of blocks of one row).  Inside a CTA three
//    kinds of warps run side by side with no CTA-wide barrier after set-up:
//    a producer warp moves blocks HBM -> shared memory with cp.async.bulk into
//    a ring of stages (a few blocks each, signalled by an mbarrier with an
//    expected byte count); filter warps test every element and append
//    survivors to a shared-memory inbox ring; selector warps keep the tray,
//    the kept list and the threshold, build the visiting orders and finish
//    each piece.  Loads keep streaming -- across piece boundaries too --
//    while the selectors sort.
//  * Two plans.  Short batches of full-length rows: a persistent grid of one
//    CTA per SM, each owning an equal share of the batch's blocks laid end to
//    end, so every SM streams the same number of bytes; rows that straddle a
//    share boundary are split.  Otherwise: one CTA per row, or per row segment
//    when a short batch of variable-length rows needs more CTAs.
//  * Every element becomes the 64-bit word (order key << 32) | ~index.  The
//    order key is the usual monotone map of float bits, so word order is value
//    order with ties broken towards the smaller index, and one 64-bit compare
//    decides every question exactly.  (The packed 64-bit words of DeepSeek
//    V4.1 Flash, kernelbench model page, entry "Single-launch CUDA bitonic
//    selection"; the ~index half gives the smaller-index tie rule.)
//  * The per-element test first runs as one float compare that can only let
//    too much through (it passes NaN and values equal to the threshold's); the
//    exact word compare runs only for element slots some lane of the warp
//    flagged (found with one warp OR-reduction).
//  * Survivors are compacted with __ballot_sync masks and __popc prefixes; one
//    shared-memory atomicAdd per warp and stage reserves inbox space.  An
//    empty inbox slot holds the word 0, which no element packs to, so the
//    selectors can tell a reserved slot whose word has not landed yet.
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
//    end of piece) gives up after a fixed number of polls, setting a status
//    bit; after one wait has given up the others poll once and the CTA drains.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "device_util.cuh"
#include "topk_select.h"

namespace topk {
namespace {

constexpr int kBlock = 1024;          // elements per block ("blocks of 1,024")
constexpr int kPermChunk = 1024;      // blocks shuffled together
constexpr int kTrayMark = 2048;       // tray words that trigger the tray sort
constexpr int kPruneStep = 512;       // new tray words that trigger a prune
constexpr int kSelectSlack = 256;     // extra words a pruned tray may keep
constexpr int kWarmElems = 8192;      // warm start: the first 32 KB of each piece
constexpr int kMaxSplit = 64;
constexpr uint32_t kWaitLimit = 1u << 22;  // polls before a wait gives up

// Launch plan, tuned for GB300's 152 SMs (results never depend on it).
constexpr int kSms = 152;
constexpr int kMaxFlatCtas = 256;     // persistent grid cap (workspace slots)
constexpr int kMinFlatBlocks = 32;    // at least 128 KB per persistent CTA
constexpr int kMinSegBlocks = 32;     // at least 128 KB per split segment
constexpr int kManyRows = kSms;       // rows per call from which each gets a CTA

constexpr uint64_t kDefaultSeed = 0x5EEDC0DE1234ABCDull;

// CTA shapes: filter warps, selector warps, blocks per ring stage, ring
// stages, CTAs per SM to fit registers for, inbox and tray capacities (words).
template <int NF_, int NS_, int BPS_, int NSTAGE_, int MINB_, int INBOX_, int TRAY_>
struct Shape {
  static constexpr int NF = NF_;
  static constexpr int NS = NS_;
  static constexpr int BPS = BPS_;
  static constexpr int NSTAGE = NSTAGE_;
  static constexpr int MIN_BLOCKS = MINB_;
  static constexpr int INBOX = INBOX_;
  static constexpr int TRAY = TRAY_;
  static constexpr int NFT = NF * 32;               // filter threads
  static constexpr int NST = NS * 32;               // selector threads
  static constexpr int NTHREADS = NFT + NST + 32;   // plus the producer warp
  static constexpr int PRODUCER_WARP = NF + NS;
  static constexpr int STAGE_FLOATS = BPS * kBlock;
  static constexpr int EPT = STAGE_FLOATS / NFT;    // elements per filter thread per stage
  static constexpr int F4 = EPT / 4;                // float4 loads per filter thread per stage
  // Inbox words the selectors move per step.  A take must never reach a slot
  // reserved by a filter warp that is itself waiting for room, so it stays at
  // least one warp-stage reservation (32 * EPT words) short of the ring size.
  static constexpr int TAKE_MAX =
      (INBOX - 32 * EPT) < 1024 ? (INBOX - 32 * EPT) : 1024;
  static_assert(EPT % 4 == 0 && EPT <= 32, "whole float4s, candidate bits in one word");
  static_assert((INBOX & (INBOX - 1)) == 0, "inbox ring size is a power of two");
  static_assert(TAKE_MAX >= 256, "inbox leaves room for a take");
  static_assert(TRAY >= kTrayMark + 512 && TRAY >= TAKE_MAX, "tray holds a take past its mark");
};

using BigShape = Shape<8, 8, 4, 8, 1, 4096, 3072>;    // 544 threads, 128 KB ring, 1 CTA/SM
using SmallShape = Shape<4, 4, 1, 8, 2, 1024, 2560>;  // 288 threads, 32 KB ring

constexpr uint32_t kNoBlock = 0xFFFFFFFFu;  // descriptor of an empty stage slot

// Plans.
constexpr int kPlanRows = 0;   // CTA = (row, segment)
constexpr int kPlanFlat = 1;   // CTA = equal share of the batch's blocks

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)              header: u32 status
//   tickets   u32[rows]   split-row leader election, zero between calls
//   survivors u32[rows]   tray words that entered a bitonic tray sort, per row
//   sorts     u32[rows]   bitonic tray sorts per row
//   admitted  u32[rows]   elements that passed the threshold test, per row
//                         (the three counters accumulate until read)
//   theta     u64[rows]   split rows: best threshold word any of the row's CTAs
//                         has reached, zero between calls
//   partials  u64[slots][kp]  local top-k lists of split rows; slots =
//                         max(rows * split, 2 * kMaxFlatCtas) when rows can
//                         be split, else none
struct WsLayout {
  size_t tickets, survivors, sorts, admitted, theta, partials, total;
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

int32_t auto_split(int32_t rows, int64_t n) {
  if (rows <= 0 || rows >= kManyRows) return 1;
  const int64_t m = (n + kBlock - 1) / kBlock;
  int64_t s = kSms / rows;
  const int64_t by_len = m / kMinSegBlocks;
  if (s > by_len) s = by_len;
  if (s > kMaxSplit) s = kMaxSplit;
  if (s < 1) s = 1;
  return int32_t(s);
}

// Partial-list slots a call may need.  With the automatic plan a short batch
// may run either plan (the choice depends on whether lengths are passed).
size_t partial_slots(int32_t rows, int32_t split_arg, int32_t split) {
  size_t slots = split > 1 ? size_t(rows) * size_t(split) : 0;
  if (split_arg == 0 && rows > 0 && rows < kManyRows) {
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
  L.theta = off;
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
  int32_t kp;          // next power of two >= k: kept-list capacity
  int32_t plan;        // kPlanRows or kPlanFlat
  int32_t split;       // kPlanRows: CTAs per row
  int32_t seg_blocks;  // kPlanRows: blocks per segment
  int32_t m_full;      // blocks per full row
  float* out_vals;
  int32_t* out_idx;
  uint32_t* status;
  uint32_t* tickets;
  uint32_t* survivors;
  uint32_t* sorts;
  uint32_t* admitted;
  unsigned long long* row_theta;
  uint64_t* partials;
  uint32_t seed_lo, seed_hi;
  uint32_t flags;
};

struct SmemLayout {
  int ring, desc, inbox, tray, kept, perm, hist, bars, total;
};

template <class S>
__host__ __device__ inline SmemLayout smem_layout(int kp) {
  SmemLayout L;
  int off = 0;
  L.ring = off;
  off += S::NSTAGE * S::STAGE_FLOATS * int(sizeof(float));
  L.desc = off;
  off += S::NSTAGE * S::BPS * int(sizeof(uint32_t));
  off = (off + 15) & ~15;
  L.inbox = off;  // inbox and tray are contiguous: the leader merge uses both
  off += S::INBOX * int(sizeof(uint64_t));
  L.tray = off;
  off += S::TRAY * int(sizeof(uint64_t));
  L.kept = off;
  off += kp * int(sizeof(uint64_t));
  L.perm = off;
  off += 2 * kPermChunk * int(sizeof(uint32_t));
  L.hist = off;
  off += 256 * int(sizeof(uint32_t));
  L.bars = off;
  off += (2 * S::NSTAGE + 2) * int(sizeof(uint64_t));
  L.total = off;
  return L;
}

struct CtaState {
  uint32_t head;      // inbox: next word the selectors take
  uint32_t tail;      // inbox: next word a filter warp reserves
  int fdone;          // filter warps done with the current piece
  int piece_gen;      // pieces the selectors have finished
  int prod_chunk;     // chunk the producer is streaming
  int flags;          // selector broadcast scratch
  int cnt2;           // compaction counter
  int leader;         // this CTA drew the last ticket
  int sel_b, sel_above, sel_binc;  // histogram select: chosen bin and counts
  int sel_n, sel_done;             // selector step: words to take, piece done
  uint64_t theta;     // the threshold word the filters test against
};

// A piece: blocks [b_begin, b_end) of row r, processed with one tray.
struct Piece {
  int32_t r;
  int32_t b_begin, b_end;
  int32_t m;             // blocks in the row
  uint32_t L;            // valid length of the row
  int32_t contributors;  // CTAs sharing the row (1 = unsplit)
  int32_t slot;          // partial slot when split
  int32_t first_cta;     // kPlanFlat: first CTA of the row
};

// Cursor over a CTA's chunks (at most kPermChunk blocks of one piece).
struct Cursor {
  bool valid;
  int32_t pi;       // piece index within the CTA
  Piece pc;
  int32_t cb;       // first block of the chunk (row-local)
  int32_t cs;       // blocks in the chunk
};

__device__ __forceinline__ int64_t flat_lo(int64_t g, int64_t M, int64_t G) { return g * M / G; }
__device__ __forceinline__ int32_t flat_cta_of(int64_t b, int64_t M, int64_t G) {
  return int32_t(((b + 1) * G - 1) / M);
}

// The pi-th piece of this CTA, or false when there is none.
__device__ bool get_piece(const Params& p, int32_t pi, Piece& out) {
  const uint32_t cta = blockIdx.x;
  if (p.plan == kPlanRows) {
    if (pi != 0) return false;
    const int32_t r = int32_t(cta / uint32_t(p.split));
    const int32_t s = int32_t(cta % uint32_t(p.split));
    int64_t L = p.lengths ? int64_t(p.lengths[r]) : p.n;
    if (L < 0) L = 0;
    if (L > p.n) L = p.n;
    const int32_t m = int32_t((L + kBlock - 1) / kBlock);
    const int32_t contributors = m == 0 ? 1 : (m + p.seg_blocks - 1) / p.seg_blocks;
    if (s >= contributors) return false;
    out.r = r;
    out.m = m;
    out.L = uint32_t(L);
    out.b_begin = s * p.seg_blocks;
    out.b_end = m == 0 ? 0 : min(m, out.b_begin + p.seg_blocks);
    out.contributors = contributors;
    out.slot = r * p.split + s;
    out.first_cta = 0;
    return true;
  }
  const int64_t M = int64_t(p.rows) * p.m_full;
  const int64_t G = gridDim.x;
  const int64_t lo = flat_lo(cta, M, G), hi = flat_lo(cta + 1, M, G);
  const int64_t r0 = lo / p.m_full;
  const int64_t r = r0 + pi;
  const int64_t rs = r * p.m_full;
  if (r >= p.rows || rs >= hi) return false;
  out.r = int32_t(r);
  out.m = p.m_full;
  out.L = uint32_t(p.n);
  out.b_begin = int32_t(lo > rs ? lo - rs : 0);
  out.b_end = int32_t(hi - rs < p.m_full ? hi - rs : p.m_full);
  const int32_t g0 = flat_cta_of(rs, M, G), g1 = flat_cta_of(rs + p.m_full - 1, M, G);
  out.contributors = g1 - g0 + 1;
  out.first_cta = g0;
  out.slot = 2 * int32_t(cta) + (r == r0 ? 0 : 1);
  return true;
}

__device__ void cursor_first(const Params& p, Cursor& c) {
  c.pi = 0;
  c.valid = get_piece(p, 0, c.pc);
  c.cb = c.valid ? c.pc.b_begin : 0;
  c.cs = c.valid ? min(c.pc.b_end - c.pc.b_begin, kPermChunk) : 0;
}

__device__ void cursor_next(const Params& p, Cursor& c) {
  c.cb += c.cs;
  if (c.cb >= c.pc.b_end) {
    c.pi += 1;
    c.valid = get_piece(p, c.pi, c.pc);
    if (!c.valid) return;
    c.cb = c.pc.b_begin;
  }
  c.cs = min(c.pc.b_end - c.cb, kPermChunk);
}

// Visiting order of `cs` consecutive blocks of row `row` starting at block
// `first`: the blocks sorted by a Philox draw with the low 10 bits replaced by
// the block's position, so the order is a permutation no matter the draws and
// never depends on the scores.  perm[p] & 1023 = position visited p-th.
template <class T>
__device__ void build_visit_order(uint32_t* perm, int cs, int64_t first, int32_t row,
                                  uint32_t seed_lo, uint32_t seed_hi, bool identity, int t) {
  const int p2 = next_pow2_dev(cs);
  for (int j = t; j < p2; j += T::size) {
    uint32_t key = 0xFFFFFFFFu;
    if (j < cs) {
      if (identity) {
        key = uint32_t(j);
      } else {
        const uint4 r = philox4x32_10(make_uint4(uint32_t(first + j), uint32_t(row), 0u, 0u),
                                      seed_lo, seed_hi);
        key = (r.x & ~1023u) | uint32_t(j);
      }
    }
    perm[j] = key;
  }
  T::sync();
  bitonic_network<T, uint32_t, false>(perm, p2, 2, 1, 0, t);
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
  bitonic_network<T, uint64_t, true>(kept, kp, kp, 1, 0, t);
}

__device__ __forceinline__ void write_row(const Params& p, int32_t r, const uint64_t* kept, int t,
                                          int nt) {
  float* ov = p.out_vals + int64_t(r) * p.k;
  int32_t* oi = p.out_idx + int64_t(r) * p.k;
  for (int j = t; j < p.k; j += nt) {
    const uint64_t w = kept[j];
    if (w == 0ull) {
      ov[j] = -__int_as_float(0x7F800000);
      oi[j] = -1;
    } else {
      ov[j] = key_to_float(uint32_t(w >> 32));
      oi[j] = int32_t(~uint32_t(w));
    }
  }
}

// ---------------------------------------------------------------------------
// The selection kernel.
//
// Roles inside a CTA (no CTA-wide barrier after set-up):
//  * the producer warp (lane 0) streams each stage's blocks with
//    cp.async.bulk and writes the stage's block descriptors;
//  * NF filter warps test every element against the current threshold and
//    append survivors to a shared-memory inbox ring (empty slots hold the
//    word 0, which no element ever packs to, so a reader can tell a slot that
//    is reserved but not yet written);
//  * NS selector warps drain the inbox into the tray, raise the threshold
//    (histogram select + prune), run the bitonic tray sort when the tray
//    passes its mark, build the visiting orders and finish each piece.

template <class S>
__global__ void __launch_bounds__(S::NTHREADS, S::MIN_BLOCKS) topk_select_kernel(const Params p) {
  using Sel = Team<S::NST, 1>;
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout sl = smem_layout<S>(p.kp);
  float* ring = reinterpret_cast<float*>(smem + sl.ring);
  uint32_t* desc = reinterpret_cast<uint32_t*>(smem + sl.desc);
  uint64_t* inbox = reinterpret_cast<uint64_t*>(smem + sl.inbox);
  uint64_t* tray = reinterpret_cast<uint64_t*>(smem + sl.tray);
  uint64_t* kept = reinterpret_cast<uint64_t*>(smem + sl.kept);
  uint32_t* perm = reinterpret_cast<uint32_t*>(smem + sl.perm);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + sl.hist);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sl.bars);
  uint64_t* empty = full + S::NSTAGE;
  uint64_t* perm_ready = empty + S::NSTAGE;
  __shared__ CtaState st;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool identity = (p.flags & TOPK_FLAG_IDENTITY_ORDER) != 0;
  const int kp = p.kp, k = p.k;

  // a1: lengths outside [0, n] are clamped and reported once per row.
  if (p.plan == kPlanRows && p.lengths && tid == 0 && blockIdx.x % uint32_t(p.split) == 0) {
    const int32_t L = p.lengths[blockIdx.x / uint32_t(p.split)];
    if (L < 0 || int64_t(L) > p.n) atomicOr(p.status, TOPK_STATUS_BAD_LENGTH);
  }

  Cursor first;
  cursor_first(p, first);
  if (!first.valid) return;  // nothing for this CTA (a short row's spare segment)
  if (first.pc.m == 0) {     // a row of length 0: all padding
    for (int j = tid; j < kp; j += S::NTHREADS) kept[j] = 0ull;
    __syncthreads();
    write_row(p, first.pc.r, kept, tid, S::NTHREADS);
    return;
  }

  for (int j = tid; j < kp; j += S::NTHREADS) kept[j] = 0ull;
  for (int j = tid; j < S::INBOX; j += S::NTHREADS) inbox[j] = 0ull;
  if (tid == 0) {
    st.head = 0;
    st.tail = 0;
    st.fdone = 0;
    st.piece_gen = 0;
    st.prod_chunk = -1;
    st.theta = 0ull;
    st.flags = 0;
    for (int i = 0; i < S::NSTAGE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], S::NF);
    }
    mbar_init(&perm_ready[0], 1);
    mbar_init(&perm_ready[1], 1);
    mbar_init_fence();
  }
  __syncthreads();

  // ---------------- producer: a3, the bulk-copy stream ----------------
  if (warp == S::PRODUCER_WARP) {
    if (lane != 0) return;
    bool gave_up = false;
    uint32_t g = 0;
    Cursor cur = first;
    for (int c = 0; cur.valid; ++c, cursor_next(p, cur)) {
      const uint32_t* pc = perm + (c & 1) * kPermChunk;
      const float* row = p.scores + int64_t(cur.pc.r) * p.row_stride;
      const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
      if (!mbar_wait(&perm_ready[c & 1], (c >> 1) & 1, gave_up ? 1u : kWaitLimit)) gave_up = true;
      // the buffer of chunk c - 1 is no longer read: the selectors may refill it
      *reinterpret_cast<volatile int*>(&st.prod_chunk) = c;
      for (int i = 0; i < cur.cs; i += S::BPS, ++g) {
        const uint32_t stage = g % S::NSTAGE;
        if (g >= uint32_t(S::NSTAGE) &&
            !mbar_wait(&empty[stage], ((g / S::NSTAGE) - 1) & 1, gave_up ? 1u : kWaitLimit))
          gave_up = true;
        uint32_t bytes[S::BPS];
        const float* src[S::BPS];
        uint32_t total = 0;
#pragma unroll
        for (int b = 0; b < S::BPS; ++b) {
          bytes[b] = 0;
          src[b] = row;
          uint32_t e0 = kNoBlock;
          if (i + b < cur.cs) {
            e0 = uint32_t(cur.cb + int32_t(pc[i + b] & 1023u)) * kBlock;
            if (aligned) {
              const uint32_t valid = min(uint32_t(kBlock), cur.pc.L - e0);
              bytes[b] = (valid & ~3u) * 4u;
              src[b] = row + e0;
            }
          }
          desc[stage * S::BPS + b] = e0;
          total += bytes[b];
        }
        fence_proxy_async_smem();
        if (total) {
          mbar_arrive_expect_tx(&full[stage], total);
#pragma unroll
          for (int b = 0; b < S::BPS; ++b)
            if (bytes[b])
              bulk_load(ring + stage * S::STAGE_FLOATS + b * kBlock, src[b], bytes[b],
                        &full[stage]);
        } else {
          mbar_arrive(&full[stage]);
        }
      }
    }
    if (gave_up) atomicOr(p.status, TOPK_STATUS_TIMEOUT);
    return;
  }

  // ---------------- filter warps: a4 + a5 ----------------
  if (warp < S::NF) {
    const int ft = tid;  // 0 .. NFT-1
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint64_t th = 0ull;
    float thf = threshold_float(th);
    uint32_t admitted = 0;
    bool saw_nan = false, timed_out = false;
    int gen = 0;
    uint32_t g = 0;
    // Wait until the selectors have released piece `piece` (with its warm-start
    // threshold in place), then pick up that threshold.
    auto gate = [&](int piece) {
      uint32_t it = timed_out ? kWaitLimit : 0u;
      while (*reinterpret_cast<volatile int*>(&st.piece_gen) < piece + 1) {
        if (++it > kWaitLimit) {
          timed_out = true;
          break;
        }
        __nanosleep(128);
      }
      __syncwarp();
      th = *reinterpret_cast<volatile uint64_t*>(&st.theta);
      thf = threshold_float(th);
    };
    gate(0);
    Cursor cur = first;
    for (int c = 0; cur.valid; ++c) {
      const float* row = p.scores + int64_t(cur.pc.r) * p.row_stride;
      const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
      const uint32_t L32 = cur.pc.L;
      const int cs = cur.cs;
      for (int i = 0; i < cs; i += S::BPS, ++g) {
        const uint32_t stage = g % S::NSTAGE;
        if (!mbar_wait(&full[stage], (g / S::NSTAGE) & 1, timed_out ? 1u : kWaitLimit))
          timed_out = true;
        const uint64_t nt = *reinterpret_cast<volatile uint64_t*>(&st.theta);
        if (nt != th) {
          th = nt;
          thf = threshold_float(th);
        }
        const float* src = ring + stage * S::STAGE_FLOATS;
        uint32_t e0s[S::F4];
        bool clean = aligned;
#pragma unroll
        for (int u = 0; u < S::F4; ++u) {
          const uint32_t e0 = desc[stage * S::BPS + ((ft + S::NFT * u) >> 8)];
          e0s[u] = e0;
          clean &= e0 != kNoBlock && e0 + kBlock <= L32;
        }
        float x[S::EPT];
        uint32_t cand = 0;  // bit e: element e may beat the threshold
        if (clean) {
#pragma unroll
          for (int u = 0; u < S::F4; ++u) {
            const float4 v = reinterpret_cast<const float4*>(src)[ft + S::NFT * u];
            x[4 * u + 0] = v.x;
            x[4 * u + 1] = v.y;
            x[4 * u + 2] = v.z;
            x[4 * u + 3] = v.w;
          }
          // One question per element.  The float compare passes a superset of
          // the exact survivors (equal values, NaN); the word compare decides.
#pragma unroll
          for (int e = 0; e < S::EPT; ++e) cand |= uint32_t(!(x[e] < thf)) << e;
          if (__any_sync(0xFFFFFFFFu, cand != 0u)) {
            // Each lane walks only its own flagged elements (re-read from the
            // stage, which is not released yet): exact word test, then a warp
            // prefix of the per-lane pass counts from five ballot masks and
            // __popc, one inbox reservation, and the writes.
            auto word_at = [&](int e, bool& nan) -> uint64_t {
              const int q = ft + S::NFT * (e >> 2);
              const uint32_t bits = __float_as_uint(src[q * 4 + (e & 3)]);
              nan = (bits & 0x7FFFFFFFu) > 0x7F800000u;
              const uint32_t idx = desc[stage * S::BPS + (q >> 8)] + uint32_t((q & 255) * 4 + (e & 3));
              return (uint64_t(order_key(bits)) << 32) | uint64_t(~idx);
            };
            uint32_t passm = 0;
            for (uint32_t m = cand; m; m &= m - 1u) {
              const int e = __ffs(m) - 1;
              bool nan;
              const uint64_t w = word_at(e, nan);
              saw_nan |= nan;
              if (!nan && w > th) passm |= 1u << e;
            }
            const uint32_t np = __popc(passm);
            uint32_t off = 0, total = 0;
#pragma unroll
            for (int b = 0; b < 6; ++b) {
              const uint32_t bal = __ballot_sync(0xFFFFFFFFu, (np >> b) & 1u);
              off += uint32_t(__popc(bal & lt_mask)) << b;
              total += uint32_t(__popc(bal)) << b;
            }
            if (total) {
              uint32_t pos = 0;
              if (lane == 0) {
                pos = atomicAdd(&st.tail, total);
                admitted += total;
                // wait for room: the selectors free slots by advancing head
                uint32_t it = timed_out ? kWaitLimit : 0u;
                while (pos + total - *reinterpret_cast<volatile uint32_t*>(&st.head) >
                       uint32_t(S::INBOX)) {
                  if (++it > kWaitLimit) {
                    timed_out = true;
                    break;
                  }
                  __nanosleep(64);
                }
              }
              pos = __shfl_sync(0xFFFFFFFFu, pos, 0) + off;
              for (uint32_t m = passm; m; m &= m - 1u) {
                bool nan;
                const uint64_t w = word_at(__ffs(m) - 1, nan);
                reinterpret_cast<volatile uint64_t*>(inbox)[pos & (S::INBOX - 1)] = w;
                ++pos;
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
        } else {
#pragma unroll
          for (int u = 0; u < S::F4; ++u) {
            const int q = ft + S::NFT * u;
            const int b = q >> 8;
            const uint32_t j0 = uint32_t((q & 255) * 4);
            const uint32_t e0 = e0s[u];
            uint32_t valid = 0, copied = 0;
            if (e0 != kNoBlock) {
              valid = min(uint32_t(kBlock), L32 - e0);
              copied = aligned ? (valid & ~3u) : 0u;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t j = j0 + uint32_t(e);
              float v = 0.f;
              if (j < copied) v = src[b * kBlock + j];
              else if (j < valid) v = __ldg(row + e0 + j);
              x[4 * u + e] = v;
              if (j < valid) cand |= uint32_t(!(v < thf)) << (4 * u + e);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
        }

        const uint32_t wcand = clean ? 0u : __reduce_or_sync(0xFFFFFFFFu, cand);
        if (wcand) {
          // Stages with ragged or unaligned blocks (values partly read from
          // global memory): for each element slot some lane flagged, the exact
          // word test and a ballot mask; then one inbox reservation for the
          // warp and the writes at __popc prefix offsets.
          uint32_t pm[S::EPT];
          int total = 0;
#pragma unroll
          for (int e = 0; e < S::EPT; ++e) {
            pm[e] = 0u;
            if ((wcand >> e) & 1u) {
              bool pass = false;
              if ((cand >> e) & 1u) {
                const uint32_t bits = __float_as_uint(x[e]);
                const bool nan = (bits & 0x7FFFFFFFu) > 0x7F800000u;
                saw_nan |= nan;
                const uint32_t idx = e0s[e >> 2] + uint32_t(((ft + S::NFT * (e >> 2)) & 255) * 4 + (e & 3));
                const uint64_t w = (uint64_t(order_key(bits)) << 32) | uint64_t(~idx);
                pass = !nan && w > th;
              }
              pm[e] = __ballot_sync(0xFFFFFFFFu, pass);
              total += __popc(pm[e]);
            }
          }
          if (total) {
            uint32_t pos = 0;
            if (lane == 0) {
              pos = atomicAdd(&st.tail, uint32_t(total));
              admitted += uint32_t(total);
              // wait for room: the selectors free slots by advancing head
              uint32_t it = timed_out ? kWaitLimit : 0u;
              while (pos + uint32_t(total) - *reinterpret_cast<volatile uint32_t*>(&st.head) >
                     uint32_t(S::INBOX)) {
                if (++it > kWaitLimit) {
                  timed_out = true;
                  break;
                }
                __nanosleep(64);
              }
            }
            pos = __shfl_sync(0xFFFFFFFFu, pos, 0);
#pragma unroll
            for (int e = 0; e < S::EPT; ++e) {
              if (pm[e]) {
                if ((pm[e] >> lane) & 1u) {
                  const uint32_t bits = __float_as_uint(x[e]);
                  const uint32_t idx = e0s[e >> 2] + uint32_t(((ft + S::NFT * (e >> 2)) & 255) * 4 + (e & 3));
                  const uint64_t w = (uint64_t(order_key(bits)) << 32) | uint64_t(~idx);
                  reinterpret_cast<volatile uint64_t*>(inbox)[(pos + __popc(pm[e] & lt_mask)) &
                                                              (S::INBOX - 1)] = w;
                }
                pos += __popc(pm[e]);
              }
            }
          }
        }
      }
      Cursor nxt = cur;
      cursor_next(p, nxt);
      if (!nxt.valid || nxt.pi != cur.pi) {
        // end of a piece: report, then wait until the selectors have finished
        // it and set the next piece's warm-start threshold
        __syncwarp();
        if (lane == 0) {
          if (admitted) atomicAdd(&p.admitted[cur.pc.r], admitted);
          __threadfence_block();
          atomicAdd(&st.fdone, 1);
        }
        admitted = 0;
        ++gen;
        if (nxt.valid) gate(gen);
      }
      cur = nxt;
    }
    saw_nan = __any_sync(0xFFFFFFFFu, saw_nan);
    timed_out = __any_sync(0xFFFFFFFFu, timed_out);
    if (lane == 0) {
      if (saw_nan) atomicOr(p.status, TOPK_STATUS_NAN);
      if (timed_out) atomicOr(p.status, TOPK_STATUS_TIMEOUT);
    }
    return;
  }

  // ---------------- selector warps: a2, a6, a7, a8 ----------------
  const int stt = tid - S::NFT;  // 0 .. NST-1
  const int swarp = stt >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  bool timed_out = false;
  uint32_t nsorts = 0, nsorted = 0;
  int tray_n = 0;       // words in the tray
  int kept_n = 0;       // real words in the kept list
  int pruned = 0;       // tray words left by the last prune
  uint64_t theta = 0ull;
  uint32_t head = 0;

  // a2: visiting orders are built ahead of the producer, one chunk at a time
  Cursor bcur = first;
  int built = 0;
  auto build_next = [&]() {
    uint32_t* pb = perm + (built & 1) * kPermChunk;
    build_visit_order<Sel>(pb, bcur.cs, bcur.cb, bcur.pc.r, p.seed_lo, p.seed_hi, identity, stt);
    if (stt == 0) mbar_arrive(&perm_ready[built & 1]);
    ++built;
    cursor_next(p, bcur);
  };
  build_next();

  // Publish a threshold to the filters (and to the row's other CTAs).
  auto raise_theta = [&](uint64_t nth, const Piece& pc) {
    if (nth <= theta) return;
    theta = nth;
    if (stt == 0) {
      if (pc.contributors > 1) {
        const unsigned long long old = atomicMax(&p.row_theta[pc.r], (unsigned long long)nth);
        if (old > nth) theta = old;
      }
      *reinterpret_cast<volatile uint64_t*>(&st.theta) = theta;
    }
  };

  // a6: the tray.  A byte-wise histogram select over kept + tray finds a word
  // prefix T such that at least k words are >= T and at most kp + slack are;
  // tray words below T can never reach the best k and are dropped, and the
  // threshold rises to T.  With `sort` (the tray has passed its mark, or the
  // piece is done) the rest are bitonic-sorted and merged into the kept
  // list, whose k-th word becomes the threshold, and the tray is emptied.
  auto process_tray = [&](bool sort, const Piece& pc) {
    const int slack = kp >= kTrayMark ? 0 : kSelectSlack;
    uint64_t T = 0ull;
    if (kept_n + tray_n > kp + slack) {
      uint64_t prefix = 0ull;
      uint32_t need = uint32_t(k), greater = 0;
      for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        const uint64_t hmask = pass == 0 ? 0ull : (~0ull << (shift + 8));
        for (int b = stt; b < 256; b += S::NST) hist[b] = 0u;
        Sel::sync();
        for (int j = stt; j < kp + tray_n; j += S::NST) {
          const uint64_t w = j < kp ? kept[j] : tray[j - kp];
          if (w != 0ull && (w & hmask) == prefix) atomicAdd(&hist[(w >> shift) & 0xFFu], 1u);
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
        if (greater + binc <= uint32_t(kp + slack) || pass == 7) {
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
    for (int base0 = 0; base0 < tray_n; base0 += R * S::NST) {
      uint64_t w[R];
      bool keep[R];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const int t = base0 + u * S::NST + stt;
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
          if (keep[u]) tray[at + __popc(mask & lt_mask)] = w[u];
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
    // the bitonic tray sort: sort the r survivors and merge them in
    const int P = next_pow2_dev(max(r, 1));
    for (int t = r + stt; t < P; t += S::NST) tray[t] = 0ull;
    Sel::sync();
    bitonic_network<Sel, uint64_t, true>(tray, P, 2, 1, 0, stt);
    merge_into_kept<Sel>(kept, tray, P, kp, stt);
    ++nsorts;
    nsorted += uint32_t(r);
    kept_n = min(kp, kept_n + r);
    tray_n = 0;
    pruned = 0;
    raise_theta(kept[k - 1], pc);
  };

  // Move up to `n` reserved inbox words into the tray (a slot still 0 is
  // reserved but not yet written: wait for it), and free their slots.
  auto take = [&](int n) {
    for (int j = stt; j < n; j += S::NST) {
      volatile uint64_t* slot =
          reinterpret_cast<volatile uint64_t*>(inbox) + ((head + uint32_t(j)) & (S::INBOX - 1));
      uint64_t w = *slot;
      uint32_t it = timed_out ? kWaitLimit : 0u;
      while (w == 0ull) {
        if (++it > kWaitLimit) {
          timed_out = true;
          break;
        }
        __nanosleep(32);
        w = *slot;
      }
      *slot = 0ull;
      tray[tray_n + j] = w;
    }
    __threadfence_block();  // the emptied slots are visible before head moves
    Sel::sync();
    head += uint32_t(n);
    tray_n += n;
    if (stt == 0) *reinterpret_cast<volatile uint32_t*>(&st.head) = head;
  };

  // Warm start: before the filters see a piece, take a threshold from its
  // first 32 KB (the first stages of its first chunk, read where they sit in
  // the ring -- the filters are held back, so the producer cannot reuse those
  // stages yet).  A key prefix T with at least k of those elements at or above
  // it bounds the piece's k-th largest from below, so every filter starts with
  // a working threshold instead of -inf.
  auto warm_start = [&](const Cursor& cu, uint32_t g0, int chunk, const Piece& pc) {
    // The producer needs this chunk's visiting order before it can fill the
    // stages waited on below.  It has finished every chunk before this one
    // (the filters completed them), so the order's buffer is free.
    if (bcur.valid && built <= chunk) build_next();
    const int nst = min((kWarmElems + S::STAGE_FLOATS - 1) / S::STAGE_FLOATS,
                        (cu.cs + S::BPS - 1) / S::BPS);
    for (int sidx = 0; sidx < nst; ++sidx) {
      const uint32_t gs = g0 + uint32_t(sidx);
      if (!mbar_wait(&full[gs % S::NSTAGE], (gs / S::NSTAGE) & 1, timed_out ? 1u : kWaitLimit))
        timed_out = true;
    }
    const float* row = p.scores + int64_t(pc.r) * p.row_stride;
    const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    // key of sample element j, or 0 for an empty slot or NaN (no valid key is 0)
    auto sample_key = [&](int j) -> uint32_t {
      const int sidx = j / S::STAGE_FLOATS;
      const int e = j - sidx * S::STAGE_FLOATS;
      const uint32_t stage = (g0 + uint32_t(sidx)) % S::NSTAGE;
      const uint32_t e0 = desc[stage * S::BPS + (e >> 10)];
      if (e0 == kNoBlock) return 0u;
      const uint32_t jj = uint32_t(e & (kBlock - 1));
      const uint32_t valid = min(uint32_t(kBlock), pc.L - e0);
      if (jj >= valid) return 0u;
      const float x = (aligned && jj < (valid & ~3u)) ? ring[stage * S::STAGE_FLOATS + e]
                                                      : __ldg(row + e0 + jj);
      const uint32_t bits = __float_as_uint(x);
      return (bits & 0x7FFFFFFFu) > 0x7F800000u ? 0u : order_key(bits);
    };
    const int total = nst * S::STAGE_FLOATS;
    if (stt == 0) st.cnt2 = 0;
    Sel::sync();
    int mine = 0;
    for (int j = stt; j < total; j += S::NST) mine += sample_key(j) != 0u;
    atomicAdd(&st.cnt2, mine);
    Sel::sync();
    if (st.cnt2 < k) return;  // too few elements to bound anything
    const int slack = kp >= kTrayMark ? 0 : kSelectSlack;
    uint32_t prefix = 0, need = uint32_t(k), greater = 0;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      const uint32_t hmask = pass == 0 ? 0u : (~0u << (shift + 8));
      for (int b = stt; b < 256; b += S::NST) hist[b] = 0u;
      Sel::sync();
      for (int j = stt; j < total; j += S::NST) {
        const uint32_t key = sample_key(j);
        if (key != 0u && (key & hmask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
      }
      Sel::sync();
      if (swarp == 0) {
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
      Sel::sync();
      prefix |= b << shift;
      greater += above;
      need -= above;
      if (greater + binc <= uint32_t(k + slack) || pass == 3) break;
    }
    // words w > (prefix << 32) - 1 are exactly the words whose key is >= prefix;
    // a zero prefix bounds nothing
    if (prefix) raise_theta((uint64_t(prefix) << 32) - 1ull, pc);
  };

  Cursor pcur = first;  // the piece being selected
  int piece_no = 0;
  uint32_t g_sel = 0;   // ring stage index where the piece starts
  int pchunk = 0;       // chunk index where the piece starts
  while (pcur.valid) {
    const Piece pc = pcur.pc;
    warm_start(pcur, g_sel, pchunk, pc);
    Sel::sync();
    if (stt == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&st.piece_gen) = piece_no + 1;  // release the filters
    }
    uint32_t idle = 0;
    for (;;) {
      // build the next visiting order once the producer no longer reads its buffer
      if (bcur.valid) {
        if (stt == 0)
          st.flags = (*reinterpret_cast<volatile int*>(&st.prod_chunk) >= built - 1) ? 1 : 0;
        Sel::sync();
        const bool go = st.flags != 0;
        Sel::sync();
        if (go) build_next();
      }
      // what is waiting: read the finished-filter count before the tail, so a
      // full count means the tail is final
      if (stt == 0) {
        const int fd = *reinterpret_cast<volatile int*>(&st.fdone);
        const uint32_t tail = *reinterpret_cast<volatile uint32_t*>(&st.tail);
        const uint32_t avail = tail - head;
        int n = int(min(avail, uint32_t(S::TRAY - tray_n)));
        if (n > S::TAKE_MAX) n = S::TAKE_MAX;
        st.sel_n = n;
        st.sel_done = (fd == S::NF && avail == 0) ? 1 : 0;
        if (pc.contributors > 1) {
          const unsigned long long gt =
              *reinterpret_cast<volatile unsigned long long*>(&p.row_theta[pc.r]);
          if (gt > theta) *reinterpret_cast<volatile uint64_t*>(&st.theta) = gt;
        }
      }
      Sel::sync();
      const int n = st.sel_n;
      const bool done = st.sel_done != 0;
      theta = *reinterpret_cast<volatile uint64_t*>(&st.theta);
      Sel::sync();
      if (done) break;
      if (n > 0) {
        idle = 0;
        take(n);
        if (tray_n >= kTrayMark) process_tray(true, pc);
        else if (tray_n >= pruned + kPruneStep) process_tray(false, pc);
      } else {
        if (++idle > kWaitLimit) {
          timed_out = true;
          break;
        }
        __nanosleep(64);
      }
    }

    // end of the piece: final sort, then the row's output (directly, or
    // through the split-row ticket)
    if (tray_n > 0) process_tray(true, pc);
    if (stt == 0) {
      atomicAdd(&p.sorts[pc.r], nsorts);
      atomicAdd(&p.survivors[pc.r], nsorted);
    }
    nsorts = 0;
    nsorted = 0;
    if (pc.contributors == 1) {
      write_row(p, pc.r, kept, stt, S::NST);
    } else {
      // a7: publish the local list, take a ticket; the last ticket merges.
      uint64_t* mine = p.partials + int64_t(pc.slot) * kp;
      for (int j = stt; j < kp; j += S::NST) mine[j] = kept[j];
      __threadfence();
      Sel::sync();
      if (stt == 0) {
        const uint32_t t = atomicAdd(&p.tickets[pc.r], 1u);
        st.leader = (t == uint32_t(pc.contributors - 1)) ? 1 : 0;
      }
      Sel::sync();
      if (st.leader) {
        __threadfence();
        // Gather lists into the idle inbox + tray and merge them as a tree of
        // parallel pairwise merges; the running result stays in slot 0.
        uint64_t* slots = inbox;  // inbox and tray are contiguous
        const int cap = (S::INBOX + S::TRAY) / kp;
        for (int j = stt; j < kp; j += S::NST) slots[j] = kept[j];
        int next_other = 0;  // next contributor to gather (never this CTA)
        const int self = p.plan == kPlanRows ? int(blockIdx.x % uint32_t(p.split))
                                             : int(blockIdx.x) - pc.first_cta;
        int remaining = pc.contributors - 1;
        while (remaining > 0) {
          const int takeq = min(remaining, cap - 1);
          int o = next_other;
          for (int q = 1; q <= takeq; ++q, ++o) {
            if (o == self) ++o;
            int64_t slot;
            if (p.plan == kPlanRows) {
              slot = int64_t(pc.r) * p.split + o;
            } else {
              const int64_t M = int64_t(p.rows) * p.m_full, G = gridDim.x;
              const int64_t go = pc.first_cta + o;
              slot = 2 * go + (flat_lo(go, M, G) / p.m_full == pc.r ? 0 : 1);
            }
            const uint64_t* other = p.partials + slot * kp;
            for (int j = stt; j < kp; j += S::NST) slots[q * kp + j] = __ldcg(other + j);
          }
          next_other = o;
          remaining -= takeq;
          Sel::sync();
          const int nl = takeq + 1;
          for (int gap = 1; gap < nl; gap <<= 1) {
            // pairs (q, q + gap) for q a multiple of 2*gap with q + gap < nl
            const int npairs = (nl - gap + 2 * gap - 1) / (2 * gap);
            for (int u = stt; u < npairs * kp; u += S::NST) {
              const int pr = u / kp, j = u - pr * kp;
              uint64_t* a = slots + (2 * gap * pr) * kp;
              const uint64_t* b = a + gap * kp;
              const uint64_t x = a[j], y = b[kp - 1 - j];
              a[j] = x > y ? x : y;
            }
            Sel::sync();
            bitonic_network<Sel, uint64_t, true>(slots, kp, kp, npairs, 2 * gap * kp, stt);
          }
        }
        write_row(p, pc.r, slots, stt, S::NST);
        Sel::sync();
        for (int j = stt; j < S::INBOX; j += S::NST) inbox[j] = 0ull;  // empty slots again
        __threadfence_block();
        if (stt == 0) {
          p.row_theta[pc.r] = 0ull;
          atomicExch(&p.tickets[pc.r], 0u);
        }
      }
    }
    // a clean tray and threshold for the next piece, then release the filters
    Sel::sync();
    for (int j = stt; j < kp; j += S::NST) kept[j] = 0ull;
    tray_n = 0;
    kept_n = 0;
    pruned = 0;
    theta = 0ull;
    // skip to the next piece
    do {
      g_sel += uint32_t((pcur.cs + S::BPS - 1) / S::BPS);
      cursor_next(p, pcur);
      ++pchunk;
    } while (pcur.valid && pcur.pi == piece_no);
    ++piece_no;
    Sel::sync();
    if (stt == 0) {
      st.fdone = 0;
      *reinterpret_cast<volatile uint64_t*>(&st.theta) = 0ull;
    }
    Sel::sync();
  }
  timed_out = Sel::sync_or(timed_out);
  if (stt == 0 && timed_out) atomicOr(p.status, TOPK_STATUS_TIMEOUT);
}

__global__ void __launch_bounds__(256)
visit_order_kernel(int32_t m, int32_t row, int64_t first, uint32_t seed_lo, uint32_t seed_hi,
                   int32_t* out) {
  __shared__ uint32_t perm[kPermChunk];
  build_visit_order<Team<256, 0>>(perm, m, first, row, seed_lo, seed_hi, false, threadIdx.x);
  for (int j = threadIdx.x; j < m; j += 256) out[j] = int32_t(perm[j] & 1023u);
}

// ---------------------------------------------------------------------------
// Host side.

struct DeviceInfo {
  std::atomic<int> configured{0};
  int sms = 0;
};
DeviceInfo g_devices[64];

cudaError_t configure_device(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  DeviceInfo* info = dev < 64 ? &g_devices[dev] : nullptr;
  if (info && info->configured.load()) {
    *sms = info->sms;
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(topk_select_kernel<BigShape>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_layout<BigShape>(TOPK_MAX_K).total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_select_kernel<SmallShape>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_layout<SmallShape>(TOPK_MAX_K).total);
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

int32_t resolve_split(int32_t rows, int64_t n, int32_t split) {
  return split == 0 ? auto_split(rows, n) : split;
}

}  // namespace
}  // namespace topk

using namespace topk;

// ---------------------------------------------------------------------------
// Workspace for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they select: code
// running inside a CUDA-graph capture that must not allocate, allocation-free
// real-time paths, plug-ins whose host framework owns every allocation and
// hands out only input and output buffers.  For them topk_select_noalloc uses
// this file-scope device array as its workspace.  Every GPU that loads this
// library keeps the array (kNoAllocWsBytes) until the process exits.  In host
// code `g_noalloc_ws` names a host-side stand-in, not device memory: its
// device address is looked up once per device with cudaGetSymbolAddress.
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
  const WsLayout wl = ws_layout(rows, next_pow2(k), partial_slots(rows, 0, resolve_split(rows, n, 0)));
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
  return auto_split(rows, n);
}

size_t topk_ws_bytes_ex(int32_t rows, int64_t n, int32_t k, int32_t split) {
  if (!shape_ok(rows, n, k) || split < 0 || split > kMaxSplit) return 0;
  const int32_t S = resolve_split(rows, n, split);
  return ws_layout(rows, next_pow2(k), partial_slots(rows, split, S)).total;
}

size_t topk_ws_bytes(int32_t rows, int64_t n, int32_t k) {
  return topk_ws_bytes_ex(rows, n, k, 0);
}

int topk_select_ex(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                   const int32_t* lengths_or_null, int32_t k, float* out_vals, int32_t* out_idx,
                   void* ws, void* stream, int32_t split, uint64_t seed, uint32_t flags) {
  if (!shape_ok(rows, n, k) || row_stride < n || split < 0 || split > kMaxSplit)
    return TOPK_ERR_SHAPE;
  if (rows == 0) return TOPK_OK;
  if (!scores || !out_vals || !out_idx) return TOPK_ERR_NULL;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return TOPK_ERR_WS;

  const int32_t S = resolve_split(rows, n, split);
  const int32_t kp = next_pow2(k);
  const WsLayout wl = ws_layout(rows, kp, partial_slots(rows, split, S));
  const int64_t m_full = (n + kBlock - 1) / kBlock;

  int sms = kSms;
  if (configure_device(&sms) != cudaSuccess) return TOPK_ERR_LAUNCH;

  unsigned char* w = static_cast<unsigned char*>(ws);
  Params p;
  p.scores = scores;
  p.row_stride = row_stride;
  p.n = n;
  p.lengths = lengths_or_null;
  p.rows = rows;
  p.k = k;
  p.kp = kp;
  p.split = S;
  p.seg_blocks = int32_t((m_full + S - 1) / S);
  p.m_full = int32_t(m_full);
  p.out_vals = out_vals;
  p.out_idx = out_idx;
  p.status = reinterpret_cast<uint32_t*>(w);
  p.tickets = reinterpret_cast<uint32_t*>(w + wl.tickets);
  p.survivors = reinterpret_cast<uint32_t*>(w + wl.survivors);
  p.sorts = reinterpret_cast<uint32_t*>(w + wl.sorts);
  p.admitted = reinterpret_cast<uint32_t*>(w + wl.admitted);
  p.row_theta = reinterpret_cast<unsigned long long*>(w + wl.theta);
  p.partials = reinterpret_cast<uint64_t*>(w + wl.partials);
  p.seed_lo = uint32_t(seed);
  p.seed_hi = uint32_t(seed >> 32);
  p.flags = flags;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool flat = split == 0 && lengths_or_null == nullptr && rows < kManyRows;
  if (flat) {
    // persistent: one CTA per SM, equal shares of the batch's blocks
    const int64_t M = int64_t(rows) * m_full;
    int64_t G = sms < kMaxFlatCtas ? sms : kMaxFlatCtas;
    const int64_t by_len = (M + kMinFlatBlocks - 1) / kMinFlatBlocks;
    if (G > by_len) G = by_len;
    if (G < 1) G = 1;
    p.plan = kPlanFlat;
    p.split = 1;
    topk_select_kernel<BigShape><<<unsigned(G), BigShape::NTHREADS,
                                   smem_layout<BigShape>(kp).total, st>>>(p);
  } else {
    const int64_t grid = int64_t(rows) * S;
    if (grid > INT32_MAX) return TOPK_ERR_SHAPE;
    p.plan = kPlanRows;
    if (S == 1 && rows >= kManyRows) {
      topk_select_kernel<SmallShape><<<unsigned(grid), SmallShape::NTHREADS,
                                       smem_layout<SmallShape>(kp).total, st>>>(p);
    } else {
      topk_select_kernel<BigShape><<<unsigned(grid), BigShape::NTHREADS,
                                     smem_layout<BigShape>(kp).total, st>>>(p);
    }
  }
  return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_LAUNCH;
}

int topk_select(const float* scores, int32_t rows, int64_t n, int64_t row_stride,
                const int32_t* lengths_or_null, int32_t k, float* out_vals, int32_t* out_idx,
                void* ws, void* stream) {
  return topk_select_ex(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx, ws,
                        stream, 0, kDefaultSeed, 0u);
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
  const int32_t S = resolve_split(rows, n, split);
  const WsLayout wl = ws_layout(rows, next_pow2(k), partial_slots(rows, split, S));
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

int topk_visit_order(int32_t m, int32_t row, int64_t first_block, uint64_t seed,
                     int32_t* order_out, void* stream) {
  if (m < 1 || m > kPermChunk || !order_out || first_block < 0) return TOPK_ERR_ARG;
  visit_order_kernel<<<1, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      m, row, first_block, uint32_t(seed), uint32_t(seed >> 32), order_out);
  return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_LAUNCH;
}

}  // extern "C"
