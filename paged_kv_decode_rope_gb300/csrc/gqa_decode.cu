// gqa_decode.cu -- paged grouped-query decode attention with split-KV and a
// log-sum-exp merge, for sm_103a.
//
// What it computes ("Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference – Start here", the direct paged decode attention item): for every
// sequence b and query head i, attention of the rotated query over the
// seq_lens[b] tokens its block table maps, with a softmax accumulated online in
// fp32, reading the pages where they lie (no contiguous copy) and never
// storing the scores. Query heads i = h*G .. h*G+G-1 share kv head h, and one
// load of a page serves all G of them. Long sequences are split across warps
// and the splits merged by their log-sum-exp (flash-decoding; not on the
// pages).
//
// Design (GB300-first, HBM bound: per token and kv head it reads 256 B; the
// G query heads of a group make the work a tiny dense contraction):
//  * Work items are (sequence, kv head, page) triples, enumerated sequence-
//    major. A persistent grid of one CTA per SM cuts the item list into equal
//    contiguous ranges, one range per warp, so long and short sequences
//    balance at page granularity with no host-side planning.
//  * Each warp streams its range through its own shared-memory ring of 2-3
//    stages: lane 0 issues one TMA tensor load per page (cp.async.bulk.tensor,
//    a 32-row box holding the head's 16 K rows then its 16 V rows, 128-byte
//    swizzle, completion counted in bytes on an mbarrier, L2 evict-first
//    since each page is read once), plus 1-D bulk copies of the G query rows
//    whenever a new (sequence, head) piece starts. No thread spends registers
//    or issue slots on global loads.
//  * Per page the warp runs two m16n8k16 bf16 tensor-core products with fp32
//    accumulation. Scores S[16 x 16 tokens] = Q K^T take Q as A with rows
//    0-7 = the G heads' q (pre-scaled by scale*log2 e) rounded to bf16 and rows
//    8-15 = the rounding remainders, so row h + row h+8 is q.k to ~2^-16
//    relative. The softmax is online per page: one max per head over its 16
//    tokens (two shuffles), exp2, one rescale of the accumulator when the max
//    grows. The score accumulator's register layout is exactly the A operand
//    of O += P V, so P goes straight from registers into the second product,
//    again as bf16 hi rows 0-7 and remainder rows 8-15. K fragments come from
//    ldmatrix, V fragments from ldmatrix.trans, conflict-free thanks to the
//    swizzle.
//  * A (sequence, head) segment that lies inside one warp range is finished
//    by that warp. A segment cut by range boundaries leaves one piece per
//    range (unnormalised accumulator, max and sum). The pieces are merged by
//    their log-sum-exp in the same kernel, after the CTA's warps have all
//    finished their ranges: pieces within the CTA through shared memory, and
//    a segment that crosses into a neighbouring CTA (at most one at each end
//    of a CTA's ranges) through workspace slots whose words say whether they
//    have been written in this call: the CTA holding the segment's last
//    pages waits (bounded) until its neighbours' partials are all there and
//    merges them, the others publish and go on. A CTA only waits for CTAs of
//    earlier groups, and no second kernel (with its launch and dependency
//    hand-off) is needed.
#include <atomic>
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kScanOffset = 512;           // scan scratch (16 ints) after the mbarriers
constexpr int kHdrBytes = 1024;            // mbarriers (<= 64 warp-stages * 8 B) + scan scratch
constexpr int kMinRangePages = 4;          // an even cut at or above this: ranges of twice it
constexpr int kSmallRangePages = 2;        // smallest automatic range, for little work
// Automatic partition weights: a page costs kPageUnits, and each (sequence,
// kv head) segment adds kSegUnits for the fixed work of its pieces (query
// rows, the new token, the merges and result stores), about 1 1/4 pages
// (measured: 3 to 8 units tried; 5 was best on the skewed batch, 30.8 -> 30.2
// us per layer, and neutral elsewhere). Without it a range of many short
// segments takes visibly longer than the others.
constexpr int kSpareSms = 4;              // SMs left without a decode CTA (see launch_decode)
constexpr int kPageUnits = 4;
constexpr int kSegUnits = 5;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kHalfDim = kHeadDim / 2;

// Kernel modes: decode with split pieces merged by the merge kernel; decode
// leaving every piece for paged_kv_split_combine; and the whole step (RoPE of
// the new token's q and k, its append into the pool, then the decode).
constexpr int kModeDecode = 0;
constexpr int kModePartials = 1;
constexpr int kModeStep = 2;

// How much of a stage's copies one issue() call starts (see the kernel).
constexpr int kIssueAll = 0;
constexpr int kIssuePage = 1;
constexpr int kIssueSide = 2;


// Each warp owns a ring of Cfg::kStages stages. A stage is a 1 KiB-aligned 4 KiB
// K/V block (one 32-row TMA box, 128-byte swizzle) plus a side buffer for the
// small rows a page may bring along: the group's fp32 q_rot rows (decode
// mode) or, in step mode, the sequence's cos/sin row (32 frequencies, each
// {cos_hi, cos_lo, sin_hi, sin_lo} in fp32), the group's raw bf16 q rows and
// the new token's raw k and v rows.
constexpr int kTrigBytes = kHalfDim * 16;  // one sequence's row of the fp32 pair table

// Warps per CTA and ring depth: three stages in flight per warp; groups of
// up to 4 heads fit 12 warps in shared memory (rings, side rings and merge
// slots), groups of 5-8 heads 10 (their registers). Measured against 16 x 2
// and 14 x 2: 12 x 3 is 0.5 us a layer faster on the batch-64 step.
template <int G>
struct Cfg {
  static constexpr int kWarps = G <= 4 ? 12 : 10;
  static constexpr int kStages = 3;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kQBytes = G * kHeadDim * 4;  // the group's fp32 query rows
  static constexpr int kStepSideBytes = kTrigBytes + G * kRowBytes + 2 * kRowBytes;
  static constexpr int kSideBytes = kQBytes > kStepSideBytes ? kQBytes : kStepSideBytes;
  static constexpr int kSlotFloats = ((G * kHeadDim + 2 * G) + 3) / 4 * 4;
};

struct DecodeParams {
  long long num_pages;
  int hkv;
  const float* q_rot;  // [batch][hq][64] (already offset to this launch's first sequence)
  float* out;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* seq_lens;
  int batch;
  int hq;
  float qscale;  // scale * log2(e): scores live in the base-2 domain
  int pages_per_split;
  float* slots;  // [group][2]: a group's partial of the segment crossing its start (0) / end (1);
                 // zero between calls
  float* o_part;
  float* lse_part;
  int32_t* num_splits;
  int max_splits;
  int* err;
  uint32_t merge_looks;  // looks of a merger at other CTAs' partials before PKV_ERR_TIMEOUT
  const int* plan;       // the workspace's plan area (automatic partition only), or null
  int plan_key;          // this launch shape's plan key
  int ring_offset;  // byte offset of the copy rings in dynamic shared memory (rounded up to 1 KiB)
  // step mode
  const uint16_t* q_raw;    // bf16 [batch][hq][64]
  const uint16_t* k_new;    // bf16 [batch][hkv][64]
  const uint16_t* v_new;    // bf16 [batch][hkv][64]
  const float4* rope_ff;    // [rope_positions][32] {cos_hi, cos_lo, sin_hi, sin_lo} (fp32 pairs)
  const double2* rope_dd;   // [rope_positions][32] {cos, sin} in fp64
  const int32_t* positions; // [batch] RoPE position of each new token
  int rope_positions;
  float* q_rot_out;         // fp32 [batch][hq][64] or null
  uint8_t* pool_w;          // the pool's bytes, for the new token's rows
};

size_t ring_offset_bytes() {
  // sequence lengths and page prefix sums
  return static_cast<size_t>(kHdrBytes) +
         ((sizeof(int) * (2 * kDecodeBatchChunk + 1) + 1023) / 1024) * 1024;
}

template <int G>
size_t smem_bytes() {
  // +1 KiB so the K/V rings can start on a 1 KiB boundary (128-byte swizzle
  // atoms); the side rings follow them.
  return ring_offset_bytes() + 1024 +
         static_cast<size_t>(Cfg<G>::kWarps) * Cfg<G>::kStages * (kHeadPageBytes + Cfg<G>::kSideBytes) +
         static_cast<size_t>(Cfg<G>::kWarps) * Cfg<G>::kSlotFloats * sizeof(float);
}

struct Cursor {
  int item, b, h, pg, np, len;
};

__device__ __forceinline__ Cursor locate(int item, const int* s_pre, const int* s_len, int batch,
                                         int hkv) {
  int lo = 0, hi = batch;  // hkv*s_pre[lo] <= item < hkv*s_pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (hkv * s_pre[mid] <= item) lo = mid; else hi = mid;
  }
  Cursor c;
  c.item = item;
  c.b = lo;
  c.np = s_pre[lo + 1] - s_pre[lo];
  const int off = item - hkv * s_pre[lo];
  c.h = off / c.np;
  c.pg = off - c.h * c.np;
  c.len = s_len[lo];
  return c;
}

// Exclusive prefix sum of pages per sequence into s_pre[0..batch], total last.
template <int kT>
__device__ void scan_pages(const int* s_len, int* s_pre, int batch, int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (batch + kT - 1) / kT;
  const int beg = min(tid * per, batch), end = min(beg + per, batch);
  int local = 0;
  for (int b = beg; b < end; ++b) local += (s_len[b] + kPage - 1) / kPage;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  // this warp's offset: the warp totals before it, summed across lanes
  int wofs = lane < warp ? s_warp[lane] : 0;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) wofs += __shfl_xor_sync(kFull, wofs, o);
  int run = wofs + incl - local;
  for (int b = beg; b < end; ++b) {
    s_pre[b] = run;
    run += (s_len[b] + kPage - 1) / kPage;
  }
  if (tid == kT - 1) s_pre[batch] = wofs + incl;
  __syncthreads();
}

// The automatic partition of a launch's work items over its warps. Work
// units are laid out segment by segment (segment s = sequence * hkv + kv
// head, its pages items P_s .. P_s + np - 1): su units of fixed cost, then pu
// units per page, so page item i of segment s starts at unit
// pu * i + su * (s + 1). Range r covers units [r cw, (r + 1) cw) and owns the
// pages that start there. pages_per_split > 0 gives plain ranges of that many
// pages (pu = 1, su = 0), as does a work list too long for 32-bit unit
// arithmetic. Short ranges cut latency when there is little work (two pages:
// more warps and SMs stream the few pages; one page was slower, four pages
// 12-14% slower on batch 8 and a single short sequence); once every warp
// would get kMinRangePages pages anyway, ranges of at least twice that keep
// the number of pieces (and merges) down.
struct Partition {
  int n_items, pu, su, total_units, cw, n_ranges;
};

__device__ __forceinline__ Partition make_partition(int total_pages, int batch, int hkv, int nwarps,
                                                    int pages_per_split) {
  Partition pt;
  pt.n_items = total_pages * hkv;
  const bool weighted = pages_per_split == 0 && pt.n_items < (1 << 28);
  pt.pu = weighted ? kPageUnits : 1;
  pt.su = weighted ? kSegUnits : 0;
  pt.total_units = pt.pu * pt.n_items + pt.su * batch * hkv;
  const int even = (pt.total_units + nwarps - 1) / nwarps;
  const int min_pages = even >= pt.pu * kMinRangePages ? 2 * kMinRangePages : kSmallRangePages;
  pt.cw = pages_per_split > 0 ? pages_per_split : max(pt.pu * min_pages, even);
  pt.n_ranges = (pt.total_units + pt.cw - 1) / pt.cw;
  return pt;
}

// First page item starting at or after unit u (n_items if none). Sequence b
// starts at unit hkv (pu s_pre[b] + su b) and each of its segments spans
// pu np + su units: find b by bisection, then the segment and page directly.
__device__ __forceinline__ int partition_item_at(const Partition& pt, int u, const int* s_pre,
                                                 int batch, int hkv) {
  if (u >= pt.total_units) return pt.n_items;
  int lo = 0, hi = batch - 1;  // largest b whose first unit is <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (hkv * (pt.pu * s_pre[mid] + pt.su * mid) <= u) lo = mid; else hi = mid - 1;
  }
  const int np = s_pre[lo + 1] - s_pre[lo];
  const int off = u - hkv * (pt.pu * s_pre[lo] + pt.su * lo);
  const int seg_units = pt.pu * np + pt.su;
  const int h = off / seg_units;
  const int within = off - h * seg_units;
  const int pg = within <= pt.su ? 0 : (within - pt.su + pt.pu - 1) / pt.pu;
  return hkv * s_pre[lo] + h * np + pg;  // pg == np: the next segment's first page
}

// A sequence's length as the decode uses it: 0 (the sequence is skipped)
// when it is outside [1, cap] or, with positions, when its RoPE position
// has no row in the table; *bad gets the error bits.
__device__ __forceinline__ int checked_length(int n, int cap, const int32_t* positions, int b,
                                              int rope_positions, int* bad) {
  int e = (n < 1 || n > cap) ? PKV_ERR_SEQ_LEN : 0;
  if (positions) {
    const int pos = positions[b];
    if (pos < 0 || pos >= rope_positions) e |= PKV_ERR_POSITION;
  }
  *bad = e;
  return e ? 0 : n;
}

// A step's work plan, kept in the decode workspace after the partial slots:
// the partition depends only on the sequence lengths (and the launch shape),
// which are the same in every layer of a step, so it is worked out once per
// step (plan_kernel) instead of by every CTA of every layer. Ints:
//   [0 .. kPlanHdr)           key (the launch shape it was made for, never 0),
//                             batch, n_items, pu, su, total_units, cw, n_ranges
//   [kPlanHdr, + batch)       the lengths as checked_length gives them
//   [.., + batch + 1)         page prefix sums
//   [.., + n_ranges + 1)      first item of each range (the last one: n_items)
// A decode that finds the key of its own launch shape and the same lengths
// takes the prefix sums and its ranges from the plan; otherwise it works
// them out itself, so a stale plan costs time, never correctness.
constexpr int kPlanHdr = 16;

// A piece of a split (sequence, kv head) segment, as one lane holds it: the
// head g8 = lane / 4 and its dims 8d + 2 tig, +1 (d = 0..7), with the running
// max (base-2 domain) and sum. fold() merges another piece into it.
struct Piece {
  float m, l;
  float2 acc[8];
  __device__ __forceinline__ void fold(float mb, float lb, const float2 (&ab)[8]) {
    const float mn = fmaxf(m, mb);
    if (mn == -INFINITY) return;  // neither side has seen a token
    const float wa = fast_exp2(m - mn), wb = fast_exp2(mb - mn);
    l = l * wa + lb * wb;
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      acc[d].x = acc[d].x * wa + ab[d].x * wb;
      acc[d].y = acc[d].y * wa + ab[d].y * wb;
    }
    m = mn;
  }
};

// Slot layout (shared memory and the workspace): the accumulator as float2
// [d][head][tig] (dims 8d + 2tig, +1 of each head: a warp's 64-bit accesses
// for one d cover consecutive words, free of bank conflicts), then G maxima,
// then G sums.
template <int G>
__device__ __forceinline__ void store_piece(float* sp, const Piece& pc, int g8, int tig) {
  if (g8 >= G) return;
  float2* acc = reinterpret_cast<float2*>(sp);
#pragma unroll
  for (int d = 0; d < 8; ++d) acc[(d * G + g8) * 4 + tig] = pc.acc[d];
  if (tig == 0) {
    sp[G * kHeadDim + g8] = pc.m;
    sp[G * kHeadDim + G + g8] = pc.l;
  }
}

// Fold the k slots at sp, sp + stride, ... (in that order) into pc, as one
// log-sum-exp combination: the maxima first, then the weighted sums, so that
// the loads of all k slots are in flight together.
template <int G>
__device__ __forceinline__ void fold_run(Piece& pc, const float* sp, int stride, int k, int g8,
                                         int tig) {
  if (k <= 0 || g8 >= G) return;
  float mx = pc.m;
  for (int j = 0; j < k; ++j) mx = fmaxf(mx, sp[j * stride + G * kHeadDim + g8]);
  if (mx == -INFINITY) return;  // no piece has seen a token
  const float w0 = fast_exp2(pc.m - mx);
  pc.l *= w0;
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    pc.acc[d].x *= w0;
    pc.acc[d].y *= w0;
  }
  for (int j = 0; j < k; ++j) {
    const float* q = sp + j * stride;
    const float wj = fast_exp2(q[G * kHeadDim + g8] - mx);
    pc.l += wj * q[G * kHeadDim + G + g8];
    const float2* acc = reinterpret_cast<const float2*>(q);
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      const float2 a = acc[(d * G + g8) * 4 + tig];
      pc.acc[d].x += wj * a.x;
      pc.acc[d].y += wj * a.y;
    }
  }
  pc.m = mx;
}

// Workspace partials of segments that cross a group boundary. A word holds
// the float's bits plus one, so that 0 (the zero-filled workspace, or a slot
// reset by its merger) means "not written in this call"; bits 0xFFFFFFFF, the
// one pattern that would wrap to 0, is a NaN that arithmetic never produces.
template <int G>
__device__ __forceinline__ void publish_piece(float* sp, const Piece& pc, int g8, int tig) {
  if (g8 >= G) return;
  uint32_t* w = reinterpret_cast<uint32_t*>(sp);
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    const int i = 2 * ((d * G + g8) * 4 + tig);
    w[i] = __float_as_uint(pc.acc[d].x) + 1u;
    w[i + 1] = __float_as_uint(pc.acc[d].y) + 1u;
  }
  if (tig == 0) {
    w[G * kHeadDim + g8] = __float_as_uint(pc.m) + 1u;
    w[G * kHeadDim + G + g8] = __float_as_uint(pc.l) + 1u;
  }
}

// Fold the partials of groups g_first .. g_last of a segment into `all`, in
// group order whichever CTA does it (so the result does not depend on which
// one does). Group grp's partial is `own`; the others are read from the
// workspace through L2. Returns whether every one of those words had been
// written (all lanes agree).
template <int G>
__device__ __forceinline__ bool gather_groups(Piece& all, const Piece& own, const float* slots,
                                              int stride, int grp, int g_first, int g_last, int g8,
                                              int tig) {
  all.m = -INFINITY;
  all.l = 0.f;
#pragma unroll
  for (int d = 0; d < 8; ++d) all.acc[d] = make_float2(0.f, 0.f);
  bool complete = true;
  if (g8 < G) {
    for (int gg = g_first; gg <= g_last; ++gg) {
      if (gg == grp) {
        all.fold(own.m, own.l, own.acc);
        continue;
      }
      const uint32_t* w = reinterpret_cast<const uint32_t*>(
          slots + static_cast<size_t>(2 * gg + (gg == g_first ? 1 : 0)) * stride);
      uint32_t raw[18];
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        const uint2 v = __ldcg(reinterpret_cast<const uint2*>(w) + (d * G + g8) * 4 + tig);
        raw[2 * d] = v.x;
        raw[2 * d + 1] = v.y;
      }
      raw[16] = __ldcg(w + G * kHeadDim + g8);
      raw[17] = __ldcg(w + G * kHeadDim + G + g8);
      float2 ab[8];
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        complete = complete && raw[2 * d] != 0u && raw[2 * d + 1] != 0u;
        ab[d] = make_float2(__uint_as_float(raw[2 * d] - 1u), __uint_as_float(raw[2 * d + 1] - 1u));
      }
      complete = complete && raw[16] != 0u && raw[17] != 0u;
      all.fold(__uint_as_float(raw[16] - 1u), __uint_as_float(raw[17] - 1u), ab);
    }
  }
  return __all_sync(kFull, complete);
}

// The first look of a CTA that has published its partial: the same fold as
// gather_groups, but the other groups' slots are first copied into shared
// memory at `stage` (this warp's page ring, idle once its range is done) by
// 16-byte asynchronous copies that are all in flight together, so that the
// look costs one round trip to L2 whatever the number of groups. Up to
// kStageSlots slots fit; a segment over more groups is looked at in batches.
// Only a word-by-word read: every word is either zero or its final value,
// so a look never folds a half-written partial.
template <int G>
__device__ __forceinline__ bool gather_groups_staged(Piece& all, const Piece& own,
                                                     const float* slots, uint32_t stage, int grp,
                                                     int g_first, int g_last, int g8, int tig,
                                                     int lane) {
  using C = Cfg<G>;
  constexpr int kChunks = C::kSlotFloats / 4;
  constexpr int kStageSlots = C::kStages * kHeadPageBytes / (C::kSlotFloats * 4);
  static_assert(kStageSlots >= 2, "the page ring holds at least two slots");
  all.m = -INFINITY;
  all.l = 0.f;
#pragma unroll
  for (int d = 0; d < 8; ++d) all.acc[d] = make_float2(0.f, 0.f);
  bool complete = true;
  for (int g0 = g_first; g0 <= g_last; g0 += kStageSlots) {
    const int g1 = min(g_last, g0 + kStageSlots - 1);
    for (int gg = g0; gg <= g1; ++gg) {
      if (gg == grp) continue;
      const float* src = slots + static_cast<size_t>(2 * gg + (gg == g_first ? 1 : 0)) * C::kSlotFloats;
      const uint32_t dst = stage + static_cast<uint32_t>((gg - g0) * C::kSlotFloats * 4);
      for (int c = lane; c < kChunks; c += 32) cp_async16(dst + 16 * c, src + 4 * c);
    }
    cp_async_wait_all();
    __syncwarp();
    if (g8 < G) {
      for (int gg = g0; gg <= g1; ++gg) {
        if (gg == grp) {
          all.fold(own.m, own.l, own.acc);
          continue;
        }
        const uint32_t w = stage + static_cast<uint32_t>((gg - g0) * C::kSlotFloats * 4);
        float2 ab[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          const uint2 v = lds64u(w + 8 * ((d * G + g8) * 4 + tig));
          complete = complete && v.x != 0u && v.y != 0u;
          ab[d] = make_float2(__uint_as_float(v.x - 1u), __uint_as_float(v.y - 1u));
        }
        const uint32_t mw = lds32(w + 4 * (G * kHeadDim + g8));
        const uint32_t lw = lds32(w + 4 * (G * kHeadDim + G + g8));
        complete = complete && mw != 0u && lw != 0u;
        all.fold(__uint_as_float(mw - 1u), __uint_as_float(lw - 1u), ab);
      }
    }
    __syncwarp();  // the stage is read before the next batch lands in it
  }
  fence_proxy_async_smem();  // the ring's next page copies come after these writes
  return __all_sync(kFull, complete);
}

template <int G>
__device__ __forceinline__ void store_output(float* out_row0, const Piece& pc, int g8, int tig) {
  if (g8 >= G) return;
  const float inv = pc.l > 0.f ? 1.f / pc.l : 0.f;
  float2* dst = reinterpret_cast<float2*>(out_row0 + g8 * kHeadDim);
#pragma unroll
  for (int d = 0; d < 8; ++d) dst[4 * d + tig] = make_float2(pc.acc[d].x * inv, pc.acc[d].y * inv);
}

// Step mode, first page of a piece: rotate the group's raw q rows at the
// sequence's position and build the mma A operand. The side buffer sS holds
// the sequence's cos/sin row (fp32 pairs) and then the raw q rows.
// Thread (g8, tig) owns dims 16s + {2tig, 2tig+1, 8+2tig, 9+2tig} of head g8,
// s = 0..3, so each rotate-half pair (d, d+32) is in one thread and it needs
// cos/sin of the 8 frequencies j in {2tig, 2tig+1, 8+2tig, 9+2tig} + {0, 16}:
// cos_hi and sin_hi (the fp32 roundings of the fp64 values) of each, read
// straight from the table row (the lanes of one tig read the same 16 bytes).
// The rotation is fp32. The piece that holds page 0 also writes the rotated
// q (before scaling) to q_rot_out.
template <int G>
__device__ __forceinline__ void rope_query(const DecodeParams& p, uint32_t sS, int bh,
                                           bool write_qrot, int g8, int tig, int lane, float qs,
                                           uint32_t (&aq)[4][4]) {
  if (g8 >= G) {
#pragma unroll
    for (int s = 0; s < 4; ++s) aq[s][0] = aq[s][1] = aq[s][2] = aq[s][3] = 0u;
    return;
  }
  float cj[8], sj[8];  // j = (q & 1) + 2 tig + 8 (q >> 1), q = 0..7
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int j = (q & 1) + 2 * tig + 8 * (q >> 1);
    const float4 t = lds128f(sS + 16 * j);  // cos_hi, cos_lo, sin_hi, sin_lo
    cj[q] = t.x;
    sj[q] = t.z;
  }
  const uint32_t sQ = sS + kTrigBytes;
  // x[s][u]: dims 16s + 2tig + {0, 1} (u = 0, 1) and 16s + 8 + 2tig + {0, 1} (u = 2, 3)
  float x[4][4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float2 a = bf16x2_to_float2(lds32(sQ + (g8 * kHeadDim + 16 * s + 2 * tig) * 2));
    const float2 b = bf16x2_to_float2(lds32(sQ + (g8 * kHeadDim + 16 * s + 8 + 2 * tig) * 2));
    x[s][0] = a.x; x[s][1] = a.y; x[s][2] = b.x; x[s][3] = b.y;
  }
  float y[4][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = (u & 1) + 2 * ((u >> 1) + 2 * s);  // frequency index of dim 16s + ...
      const float c = cj[q], sv = sj[q];
      y[s][u] = x[s][u] * c - x[s + 2][u] * sv;
      y[s + 2][u] = x[s + 2][u] * c + x[s][u] * sv;
    }
  if (write_qrot && p.q_rot_out) {
    float* qo = p.q_rot_out + (static_cast<size_t>(bh) * G + g8) * kHeadDim;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      *reinterpret_cast<float2*>(qo + 16 * s + 2 * tig) = make_float2(y[s][0], y[s][1]);
      *reinterpret_cast<float2*>(qo + 16 * s + 8 + 2 * tig) = make_float2(y[s][2], y[s][3]);
    }
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float a0 = y[s][0] * qs, a1 = y[s][1] * qs, b0 = y[s][2] * qs, b1 = y[s][3] * qs;
    const uint32_t h0 = pack_bf16x2(a0, a1), h1 = pack_bf16x2(b0, b1);
    const float2 r0 = bf16x2_to_float2(h0), r1 = bf16x2_to_float2(h1);
    aq[s][0] = h0;
    aq[s][1] = pack_bf16x2(a0 - r0.x, a1 - r0.y);
    aq[s][2] = h1;
    aq[s][3] = pack_bf16x2(b0 - r1.x, b1 - r1.y);
  }
}

// Step mode, the sequence's last page: lane j rotates the pair (j, j+32) of
// the new key and copies v dims 2j, 2j+1. The rotated pair is rounded to
// bf16 exactly as fp64 arithmetic on the sequence's fp64 cos/sin rounds it
// (the bytes the append kernel stores): rotated_bf16_fast certifies the
// rounding from the fp32 pair table in the side buffer, and a lane it cannot
// certify reads the fp64 cos/sin of its frequency and rotates in fp64. Both
// rows go into the stage (128-byte swizzled, row `row`) and into the pool
// (K rows start at TMA row y, V rows at y + 16). sS is the side buffer:
// cos/sin row, then G raw q rows, then raw k and v.
template <int G>
__device__ __forceinline__ void append_new_token(const DecodeParams& p, uint32_t sK, uint32_t sV,
                                                 uint32_t sS, int pos, int y, int row, int lane) {
  const int j = lane;
  const float4 cs = lds128f(sS + 16 * j);  // cos_hi, cos_lo, sin_hi, sin_lo
  const uint32_t sKV = sS + kTrigBytes + G * kRowBytes;
  const uint16_t k0 = lds16(sKV + 2 * j), k1 = lds16(sKV + 2 * (j + kHalfDim));
  const float x0 = __uint_as_float(static_cast<uint32_t>(k0) << 16);
  const float x1 = __uint_as_float(static_cast<uint32_t>(k1) << 16);
  uint16_t y0, y1;
  const bool fast = rotated_bf16_fast(x0, x1, cs.x, cs.y, cs.z, cs.w, y0) &&
                    rotated_bf16_fast(x1, -x0, cs.x, cs.y, cs.z, cs.w, y1);
  if (!fast) {
    const double2 cd = p.rope_dd[static_cast<size_t>(pos) * kHalfDim + j];
    rotate_key_pair(k0, k1, cd.x, cd.y, y0, y1);
  }
  const uint32_t v01 = lds32(sKV + kRowBytes + 4 * j);
  auto swz = [&](int d) {
    return static_cast<uint32_t>(row * kRowBytes + (((d >> 3) ^ (row & 7)) << 4) + (d & 7) * 2);
  };
  sts16(sK + swz(j), y0);
  sts16(sK + swz(j + kHalfDim), y1);
  sts32(sV + swz(2 * j), v01);
  uint8_t* krow = p.pool_w + (static_cast<size_t>(y) + row) * kRowBytes;
  uint8_t* vrow = p.pool_w + (static_cast<size_t>(y) + kPage + row) * kRowBytes;
  reinterpret_cast<uint16_t*>(krow)[j] = y0;
  reinterpret_cast<uint16_t*>(krow)[j + kHalfDim] = y1;
  reinterpret_cast<uint32_t*>(vrow)[j] = v01;
}

template <int G, int kMode>
__global__ void __launch_bounds__(Cfg<G>::kThreads, 1)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  using C = Cfg<G>;
  constexpr bool kPartials = kMode == kModePartials;
  constexpr bool kStep = kMode == kModeStep;
  constexpr int kW = C::kWarps;
  constexpr int kT = C::kThreads;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2;                 // mma row group: head g8 (rows g8 and g8+8)
  const int tig = lane & 3;                 // thread in group
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: which matrix / which row this lane addresses
  int* s_warp = reinterpret_cast<int*>(smem + kScanOffset);
  int* s_len = reinterpret_cast<int*>(smem + kHdrBytes);
  int* s_pre = s_len + p.batch;
  __shared__ int s_bad;  // PKV_ERR_SEQ_LEN / PKV_ERR_POSITION of sequences skipped here
  __shared__ int s_plan[kPlanHdr];
  const uint32_t bar0 = smem_addr(smem) + warp * C::kStages * 8;
  const uint32_t ring_base = (smem_addr(smem) + p.ring_offset + 1023u) & ~1023u;
  const uint32_t ring0 = ring_base + warp * C::kStages * kHeadPageBytes;
  const uint32_t side0 = ring_base + kW * C::kStages * kHeadPageBytes + warp * C::kStages * C::kSideBytes;
  const void* map = &kv_map;

  // Sequence lengths (invalid ones become empty) and the page prefix sums.
  // Everything before grid_dependency_wait() overlaps the end of the previous
  // kernel in the stream. In decode and partials mode that is shared-memory
  // set-up only. In step mode it also covers the sequence lengths, the block
  // tables and the first pages of each warp's range, which the previous
  // kernel must not write (see paged_decode_step); the step's query and new
  // token rows and all of its stores come after the wait.
  if (tid == 0) s_bad = 0;
  if (lane == 0)
    for (int s = 0; s < C::kStages; ++s) mbar_init(bar0 + 8 * s, 1);
  fence_mbar_init();
  __syncthreads();
  grid_launch_dependents();
  if (!kStep) grid_dependency_wait();
  // The lengths, and with a plan in the workspace its header, its lengths,
  // its prefix sums and the bounds of this warp's first range, all loaded in
  // one round trip; the plan is taken only if it was made for this launch
  // shape and these lengths.
  const int cap = p.max_blocks * kPage;
  const int* plan = p.plan;
  const int r_first = blockIdx.x * kW + warp;
  int agree = plan != nullptr, plan_bnd = 0;
  if (plan) {
    if (tid < kPlanHdr) s_plan[tid] = plan[tid];
    if (lane < 2) plan_bnd = plan[kPlanHdr + 2 * p.batch + 1 + r_first + lane];
    if (tid == 0) s_pre[p.batch] = plan[kPlanHdr + 2 * p.batch];
  }
  for (int b = tid; b < p.batch; b += kT) {
    int bad;
    const int n = checked_length(p.seq_lens[b], cap, kStep ? p.positions : nullptr, b,
                                 p.rope_positions, &bad);
    if (bad) atomicOr(&s_bad, bad);
    s_len[b] = n;
    if (plan) {
      if (plan[kPlanHdr + b] != n) agree = 0;
      s_pre[b] = plan[kPlanHdr + p.batch + b];
    }
  }
  agree = __syncthreads_and(agree);
  const bool planned = agree && s_plan[0] == p.plan_key && s_plan[1] == p.batch;
  if (!planned) scan_pages<kT>(s_len, s_pre, p.batch, s_warp);
  const Partition pt =
      planned ? Partition{s_plan[2], s_plan[3], s_plan[4], s_plan[5], s_plan[6], s_plan[7]}
              : make_partition(s_pre[p.batch], p.batch, p.hkv, gridDim.x * kW, p.pages_per_split);
  const int n_items = pt.n_items, pu = pt.pu, su = pt.su, cw = pt.cw, n_ranges = pt.n_ranges;
  auto item_at = [&](int u) { return partition_item_at(pt, u, s_pre, p.batch, p.hkv); };
  // Range of the unit at which segment sg's page item i starts.
  auto range_of = [&](int i, int sg) { return (pu * i + su * (sg + 1)) / cw; };
  const float qs = p.qscale;

  uint32_t phase_bits = 0;  // bit s: parity of the next completion of stage s
  int stage = 0;            // next stage to consume
  bool failed = false;

  // Work-item descriptors, 32 items per batch, lane t describing item base + t:
  //   y    TMA row of the page's first K row of its kv head (-1: bad page id)
  //   meta valid rows (bits 0-4) | first item of a piece (5) | last item of
  //        a piece (6) | bad page (7) | last page of the sequence (8) |
  //        page index within the sequence (9+)
  //   bh   sequence * hkv + kv head
  //   pos  step mode: the sequence's RoPE position (its row of the table)
  // The producer (copy issue) runs at most kStages items ahead of the consumer,
  // hence at most one batch ahead; the consumer keeps its own copy.
  int pd_base = 0, pd_y = -1, pd_meta = 0, pd_bh = 0, pd_pos = 0;
  int cd_base = 0, cd_y = -1, cd_meta = 0, cd_bh = 0, cd_pos = 0;

  auto describe = [&](int base, int i0, int i1) {
    pd_base = base;
    const int item = base + lane;
    pd_y = -1;
    pd_meta = 0;
    pd_bh = 0;
    bool bad = false;
    if (item < i1) {
      const Cursor ci = locate(item, s_pre, s_len, p.batch, p.hkv);
      const int page = __ldg(p.block_tables + static_cast<size_t>(ci.b) * p.max_blocks + ci.pg);
      if (kStep) pd_pos = __ldg(p.positions + ci.b);  // checked with the lengths
      const int nv = min(kPage, ci.len - ci.pg * kPage);
      const int first = (item == i0 || ci.pg == 0) ? 1 : 0;
      const int last = (item == i1 - 1 || ci.pg == ci.np - 1) ? 1 : 0;
      bad = page < 0 || static_cast<long long>(page) >= p.num_pages;
      const int seg_last = (ci.pg == ci.np - 1) ? 1 : 0;
      pd_meta = nv | (first << 5) | (last << 6) | ((bad ? 1 : 0) << 7) | (seg_last << 8) |
                (ci.pg << 9);
      pd_bh = ci.b * p.hkv + ci.h;
      pd_y = bad ? -1 : (page * p.hkv + ci.h) * (2 * kPage);
    }
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(p.err, PKV_ERR_PAGE_ID);
  };

  // part: kIssueAll, or for the first stages of step mode kIssuePage before
  // the dependency wait (page bytes expected, no arrival) and kIssueSide after
  // it (the side rows and the stage's arrival).
  auto issue = [&](int item, int st, int i0, int i1, int part = kIssueAll) {
    if (item >= pd_base + 32) describe(pd_base + 32, i0, i1);
    const int t = item - pd_base;
    const int y = __shfl_sync(kFull, pd_y, t);
    const int meta = __shfl_sync(kFull, pd_meta, t);
    const int bh = __shfl_sync(kFull, pd_bh, t);
    const int pos = kStep ? __shfl_sync(kFull, pd_pos, t) : 0;
    if (lane == 0) {
      const bool first = (meta >> 5) & 1;
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t dst = ring0 + st * kHeadPageBytes;
      const uint32_t side = side0 + st * C::kSideBytes;
      const bool seg_last = (meta >> 8) & 1;
      const uint32_t side_bytes =
          kStep ? ((first || seg_last) ? kTrigBytes : 0u) + (first ? G * kRowBytes : 0u) +
                      (seg_last ? 2u * kRowBytes : 0u)
                : (first ? C::kQBytes : 0u);
      const uint32_t page_bytes = y < 0 ? 0u : static_cast<uint32_t>(kHeadPageBytes);
      if (part == kIssuePage) {
        if (y >= 0) {
          mbar_expect_tx(bar, page_bytes);
          tma_load_2d_hint(dst, map, 0, y, bar, l2_policy_evict_first());
        }
        return;
      }
      const uint32_t bytes = (part == kIssueSide ? 0u : page_bytes) + side_bytes;
      if (bytes == 0) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, bytes);
        if (y >= 0 && part == kIssueAll)  // the page's 16 K rows, then its 16 V rows
          tma_load_2d_hint(dst, map, 0, y, bar, l2_policy_evict_first());
        if (kStep) {
          // the sequence's cos/sin row; the group's raw q rows on a piece's
          // first page; the new token's raw k and v rows on the sequence's last
          if (first || seg_last)
            bulk_g2s(side, p.rope_ff + static_cast<size_t>(pos) * kHalfDim, kTrigBytes, bar);
          if (first)
            bulk_g2s(side + kTrigBytes, p.q_raw + static_cast<size_t>(bh) * G * kHeadDim,
                     G * kRowBytes, bar);
          if (seg_last) {
            bulk_g2s(side + kTrigBytes + G * kRowBytes, p.k_new + static_cast<size_t>(bh) * kHeadDim,
                     kRowBytes, bar);
            bulk_g2s(side + kTrigBytes + (G + 1) * kRowBytes,
                     p.v_new + static_cast<size_t>(bh) * kHeadDim, kRowBytes, bar);
          }
        } else if (first) {  // rows b*hq + h*G .. +G-1 of q_rot start at bh * G * 64
          bulk_g2s(side, p.q_rot + static_cast<size_t>(bh) * G * kHeadDim, C::kQBytes, bar);
        }
      }
    }
  };

  uint32_t aq[4][4];  // Q as the A operand, one k-step (16 dims) each: bf16 rows g8, remainders g8+8
  float o[8][4];      // O accumulator, dims 8d..8d+7: rows g8 (from P) and g8+8 (from P's remainder)
  float m_run = -INFINITY, l_run = 0.f;

  // lane 0 finds where range r starts, lane 1 where it ends (this warp's
  // first range: read from the plan when there is one)
  auto range_bounds = [&](int r, int& i0, int& i1) {
    const int i_lane = (planned && r == r_first) ? plan_bnd : item_at((r + (lane & 1)) * cw);
    i0 = __shfl_sync(kFull, i_lane, 0);
    i1 = __shfl_sync(kFull, i_lane, 1);
  };
  bool pre_issued = false;  // step mode: the first range's first pages are on their way
  if (kStep) {
    const int r = blockIdx.x * kW + warp;
    int i0 = 0, i1 = 0;
    if (r < n_ranges) range_bounds(r, i0, i1);
    if (i0 < i1) {
      describe(i0, i0, i1);
      for (int k = 0; k < C::kStages && i0 + k < i1; ++k) issue(i0 + k, k, i0, i1, kIssuePage);
      pre_issued = true;
    }
    grid_dependency_wait();
  }

  if (s_bad) {  // rows of invalid sequences: zero output (or zero split count)
    if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, s_bad);
    const int rows = p.batch * p.hq;
    for (int idx = blockIdx.x * kT + tid; idx < rows; idx += gridDim.x * kT) {
      if (s_len[idx / p.hq] != 0) continue;
      if (kPartials) {
        p.num_splits[idx] = 0;
      } else {
        if (kStep && p.q_rot_out) {
          float4* qo = reinterpret_cast<float4*>(p.q_rot_out + static_cast<size_t>(idx) * kHeadDim);
#pragma unroll
          for (int k = 0; k < kHeadDim / 4; ++k) qo[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float4* o = reinterpret_cast<float4*>(p.out + static_cast<size_t>(idx) * kHeadDim);
#pragma unroll
        for (int k = 0; k < kHeadDim / 4; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  if (n_items == 0) return;

  // Ranges come in groups of kW, one range per warp of a CTA: group grp covers
  // ranges grp kW .. grp kW + kW - 1. A segment split over ranges of one group
  // is merged in shared memory when the group ends; one that crosses a group
  // boundary (at most one at each end) goes through the workspace, and the
  // CTA of its last group merges it.
  float* s_slots = reinterpret_cast<float*>(
      smem + (ring_base - smem_addr(smem)) +
      kW * C::kStages * (kHeadPageBytes + C::kSideBytes));
  __shared__ int s_first_bh[kW];  // a range's first piece, if it continues a segment: its segment
  __shared__ bool s_has_head[kW];  // a range's last piece holds page 0 of a segment that goes on
  __shared__ int2 s_cont_groups;   // groups of the first and last pages of warp 0's continued segment
  __shared__ int3 s_head[kW];      // a range's head segment and its first and last groups
  const int n_groups = (n_ranges + kW - 1) / kW;
  // Which pieces a warp merges when the group ends follows from its range
  // bounds alone (not from how far the warp got), so every merge below
  // happens even after a timeout and the workspace slots return to zero.
  // Lane 0 works it out when the range starts, while the first pages are on
  // their way: the segment the range's first piece continues (if any), and
  // the segment whose page 0 the range holds and that goes on past it.
  auto groups_of = [&](int sg) {
    const int b = sg / p.hkv;
    const int np = s_pre[b + 1] - s_pre[b];
    const int seg_start = p.hkv * s_pre[b] + (sg - b * p.hkv) * np;
    return make_int2(range_of(seg_start, sg) / kW, range_of(seg_start + np - 1, sg) / kW);
  };
  auto plan_merges = [&](int i0, int i1) {
    if (lane != 0) return;
    int first_bh = -1;
    int3 head = make_int3(-1, 0, 0);
    if (i0 < i1) {
      const Cursor c0 = locate(i0, s_pre, s_len, p.batch, p.hkv);
      if (c0.pg > 0) first_bh = c0.b * p.hkv + c0.h;
      const Cursor cl = locate(i1 - 1, s_pre, s_len, p.batch, p.hkv);
      if (i1 - 1 - cl.pg >= i0 && cl.pg < cl.np - 1) {
        head.x = cl.b * p.hkv + cl.h;
        const int2 g = groups_of(head.x);
        head.y = g.x;
        head.z = g.y;
      }
    }
    s_first_bh[warp] = first_bh;
    s_has_head[warp] = head.x >= 0;
    s_head[warp] = head;
    if (warp == 0 && first_bh >= 0) s_cont_groups = groups_of(first_bh);
  };
  for (int grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {
    const int r = grp * kW + warp;
    int i0 = 0, i1 = 0;
    if (r < n_ranges) range_bounds(r, i0, i1);
    if (!kPartials) plan_merges(i0, i1);
    if (i0 < i1 && !failed) {
    if (!pre_issued) describe(i0, i0, i1);
    cd_base = pd_base;
    cd_y = pd_y;
    cd_meta = pd_meta;
    cd_bh = pd_bh;
    cd_pos = pd_pos;
    {
      int st = stage;
      for (int k = 0; k < C::kStages && i0 + k < i1; ++k) {
        issue(i0 + k, st, i0, i1, pre_issued ? kIssueSide : kIssueAll);
        st = (st + 1 == C::kStages) ? 0 : st + 1;
      }
    }
    pre_issued = false;
    int start_pg = 0;
    bool first_in_range = true;
    for (int i = i0; i < i1; ++i) {
      const int st = stage;
      if (!mbar_wait_bounded(bar0 + 8 * st, (phase_bits >> st) & 1u)) {
        failed = true;
        break;
      }
      phase_bits ^= 1u << st;
      if (i >= cd_base + 32) {  // the producer has already described this batch
        cd_base = pd_base;
        cd_y = pd_y;
        cd_meta = pd_meta;
        cd_bh = pd_bh;
        cd_pos = pd_pos;
      }
      const int t = i - cd_base;
      const int meta = __shfl_sync(kFull, cd_meta, t);
      const int nv = meta & 31;
      const bool first = (meta >> 5) & 1;
      const bool last = (meta >> 6) & 1;
      const bool bad = (meta >> 7) & 1;
      const uint32_t sK = ring0 + st * kHeadPageBytes;
      const uint32_t sS = side0 + st * C::kSideBytes;
      const uint32_t sV = sK + kHalfBytes;
      const bool seg_last = (meta >> 8) & 1;
      if (first) {
        start_pg = meta >> 9;
        first_in_range = (i == i0);
        if (kStep) {
          rope_query<G>(p, sS, __shfl_sync(kFull, cd_bh, t), start_pg == 0, g8, tig, lane, qs, aq);
        } else {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if (g8 < G) {
            float2 x0 = lds64f(sS + (g8 * kHeadDim + 16 * s + 2 * tig) * 4);
            float2 x1 = lds64f(sS + (g8 * kHeadDim + 16 * s + 8 + 2 * tig) * 4);
            x0.x *= qs; x0.y *= qs; x1.x *= qs; x1.y *= qs;
            const uint32_t h0 = pack_bf16x2(x0.x, x0.y), h1 = pack_bf16x2(x1.x, x1.y);
            const float2 r0 = bf16x2_to_float2(h0), r1 = bf16x2_to_float2(h1);
            aq[s][0] = h0;
            aq[s][1] = pack_bf16x2(x0.x - r0.x, x0.y - r0.y);
            aq[s][2] = h1;
            aq[s][3] = pack_bf16x2(x1.x - r1.x, x1.y - r1.y);
          } else {
            aq[s][0] = aq[s][1] = aq[s][2] = aq[s][3] = 0u;
          }
        }
        }
#pragma unroll
        for (int d = 0; d < 8; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
        m_run = -INFINITY;
        l_run = 0.f;
      }
      if (kStep && seg_last && !bad) {
        // The sequence's new token is this page's last valid row: rotate its
        // key, put K and V into the stage (the copy brought the stale slot)
        // and into the pool.
        const int y = __shfl_sync(kFull, cd_y, t);
        append_new_token<G>(p, sK, sV, sS, __shfl_sync(kFull, cd_pos, t), y, nv - 1, lane);
        __syncwarp();
      }
      if (!bad) {
        // S = Q K^T for this page's 16 tokens (n-tiles j: tokens 8j..8j+7).
        uint32_t kb[2][4][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = q >> 1, s0 = 2 * (q & 1);
          const int row = 8 * j + ri, chunk = 4 * (q & 1) + mi;
          ldsm_x4(sK + row * kRowBytes + ((chunk ^ ri) << 4), kb[j][s0][0], kb[j][s0][1],
                  kb[j][s0 + 1][0], kb[j][s0 + 1][1]);
        }
        float sc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
          for (int s = 0; s < 4; ++s) mma_bf16_16816(sc[j], aq[s], kb[j][s][0], kb[j][s][1]);
        }
        // head g8, tokens 2tig, 2tig+1, 8+2tig, 9+2tig
        float sv[4] = {sc[0][0] + sc[0][2], sc[0][1] + sc[0][3], sc[1][0] + sc[1][2],
                       sc[1][1] + sc[1][3]};
        if (nv < kPage) {
          const int t0 = 2 * tig;
          if (t0 >= nv) sv[0] = -INFINITY;
          if (t0 + 1 >= nv) sv[1] = -INFINITY;
          if (t0 + 8 >= nv) sv[2] = -INFINITY;
          if (t0 + 9 >= nv) sv[3] = -INFINITY;
        }
        float pm = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
        pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 1));
        pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 2));
        const float m_new = fmaxf(m_run, pm);
        const bool grew = m_new > m_run;
        const float alpha = grew ? fast_exp2(m_run - m_new) : 1.f;
        float pr[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) pr[k] = fast_exp2(sv[k] - m_new);
        l_run = l_run * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
        m_run = m_new;
        if (__any_sync(kFull, grew)) {
#pragma unroll
          for (int d = 0; d < 8; ++d) {
            o[d][0] *= alpha; o[d][1] *= alpha; o[d][2] *= alpha; o[d][3] *= alpha;
          }
        }
        // P as the A operand: rows g8 = bf16(p), rows g8+8 = remainder.
        uint32_t ap[4];
        {
          const uint32_t h01 = pack_bf16x2(pr[0], pr[1]), h23 = pack_bf16x2(pr[2], pr[3]);
          const float2 f01 = bf16x2_to_float2(h01), f23 = bf16x2_to_float2(h23);
          ap[0] = h01;
          ap[1] = pack_bf16x2(pr[0] - f01.x, pr[1] - f01.y);
          ap[2] = h23;
          ap[3] = pack_bf16x2(pr[2] - f23.x, pr[3] - f23.y);
        }
        // O += P V (n-tiles d: dims 8d..8d+7), V fragments transposed by ldmatrix.
        uint32_t vb[8][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = 2 * q + (mi >> 1), row = 8 * (mi & 1) + ri;
          ldsm_x4_trans(sV + row * kRowBytes + ((chunk ^ ri) << 4), vb[2 * q][0], vb[2 * q][1],
                        vb[2 * q + 1][0], vb[2 * q + 1][1]);
        }
        if (nv < kPage) {  // rows past the valid tokens hold stale shared memory
          const int t0 = 2 * tig;
          const uint32_t m0 = (t0 < nv ? 0x0000ffffu : 0u) | (t0 + 1 < nv ? 0xffff0000u : 0u);
          const uint32_t m1 = (t0 + 8 < nv ? 0x0000ffffu : 0u) | (t0 + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
          for (int d = 0; d < 8; ++d) {
            vb[d][0] &= m0;
            vb[d][1] &= m1;
          }
        }
#pragma unroll
        for (int d = 0; d < 8; ++d) mma_bf16_16816(o[d], ap, vb[d][0], vb[d][1]);
      }

      // Every lane has consumed this stage (its ldmatrix results fed the mma
      // above) before lane 0 reissues it, so no proxy fence is needed. The
      // copy goes out before any piece bookkeeping, so the ring keeps streaming.
      __syncwarp();
      if (i + C::kStages < i1) issue(i + C::kStages, st, i0, i1);
      stage = (stage + 1 == C::kStages) ? 0 : stage + 1;

      if (last) {
        // Head g8's unnormalised output at dims 8d+2tig, +1; its max and sum.
        float2 of[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) of[d] = make_float2(o[d][0] + o[d][2], o[d][1] + o[d][3]);
        float lsum = l_run + __shfl_xor_sync(kFull, l_run, 1);
        lsum += __shfl_xor_sync(kFull, lsum, 2);
        const float mh = m_run;
        const bool live = g8 < G;
        const int bh = __shfl_sync(kFull, cd_bh, t);
        const int b = bh / p.hkv, h = bh - b * p.hkv;
        const int np = s_pre[b + 1] - s_pre[b];
        const int seg_start = p.hkv * s_pre[b] + h * np;
        const int r_first = range_of(seg_start, bh);
        const int pieces = range_of(seg_start + np - 1, bh) - r_first + 1;
        const size_t row0 = static_cast<size_t>(bh) * G;  // = b*hq + h*G
        const bool complete = (start_pg == 0) && ((meta >> 9) == np - 1);
        if (kPartials) {
          const int j = r - r_first;
          if (pieces > p.max_splits) {
            if (lane == 0) atomicOr(p.err, PKV_ERR_SPLITS);
          } else if (live) {
            const size_t row = row0 + g8;
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            float2* dst = reinterpret_cast<float2*>(p.o_part + (row * p.max_splits + j) * kHeadDim);
#pragma unroll
            for (int d = 0; d < 8; ++d) dst[4 * d + tig] = make_float2(of[d].x * inv, of[d].y * inv);
            if (tig == 0) {
              p.lse_part[row * p.max_splits + j] = lsum > 0.f ? (mh + __log2f(lsum)) * kLn2 : -INFINITY;
              p.num_splits[row] = pieces;
            }
          }
        } else if (complete) {
          if (live) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            float2* dst = reinterpret_cast<float2*>(p.out + (row0 + g8) * kHeadDim);
#pragma unroll
            for (int d = 0; d < 8; ++d) dst[4 * d + tig] = make_float2(of[d].x * inv, of[d].y * inv);
          }
        } else if (first_in_range) {
          // A split piece that opens the range: its unnormalised accumulator,
          // max and sum wait in this warp's shared-memory slot for the group's
          // merge. (A split piece that closes the range stays in registers.)
          Piece pc;
          pc.m = mh;
          pc.l = lsum;
#pragma unroll
          for (int d = 0; d < 8; ++d) pc.acc[d] = of[d];
          store_piece<G>(s_slots + warp * C::kSlotFloats, pc, g8, tig);
        }
      }
    }
    }  // this warp's range

    if (!kPartials) {
      __syncthreads();  // every slot and s_first_bh of the group are written

      // Merge segment sg: pc holds its piece of range grp kW + w, and the
      // pieces of the ranges after it in the group wait in their warps' slots.
      auto merge_segment = [&](int sg, Piece& pc, int w, int g_first, int g_last) {
        // the run of following warps whose first piece continues sg
        const int w2 = w + 1 + lane;
        const unsigned run = __ballot_sync(kFull, w2 < kW && s_first_bh[w2 < kW ? w2 : 0] == sg);
        const int k = __ffs(~run) - 1;
        fold_run<G>(pc, s_slots + (w + 1) * C::kSlotFloats, C::kSlotFloats, k, g8, tig);
        float* out_row0 = p.out + static_cast<size_t>(sg) * G * kHeadDim;
        if (g_first == g_last) {  // the whole segment lies in this group
          store_output<G>(out_row0, pc, g8, tig);
          return;
        }
        // The CTA of the segment's last group merges it; the CTAs of its other
        // groups leave their partials in the workspace and move on without
        // waiting. Every word of a partial says by itself whether it has been
        // written, so the merger needs no fence: it looks until every word
        // is there, folds the partials in group order and puts the slots back
        // to zero for the next call. A CTA only ever waits for groups before
        // its own, so the wait ends; it is bounded all the same.
        if (grp != g_last) {
          publish_piece<G>(p.slots + static_cast<size_t>(2 * grp + (grp == g_first ? 1 : 0)) *
                                         C::kSlotFloats,
                           pc, g8, tig);
          return;
        }
        Piece all;
        bool done = false;
        for (uint32_t look = 0; look < p.merge_looks && !done; ++look) {
          // Two or more other groups: stage them, so that their round trips
          // overlap (not in a warp that timed out: page copies may still land
          // in its ring). Only groups of 5-8 heads: their few KV heads make
          // segments long enough to span three or more CTAs, and their kernel
          // has the registers to spare; in the register-capped kernel of 1-4
          // heads the extra code cost 0.2 us per layer where it never ran.
          if constexpr (G > 4) {
            if (g_last - g_first >= 2 && !failed) {
              done = gather_groups_staged<G>(all, pc, p.slots, ring0, grp, g_first, g_last, g8,
                                             tig, lane);
              continue;
            }
          }
          done = gather_groups<G>(all, pc, p.slots, C::kSlotFloats, grp, g_first, g_last, g8, tig);
        }
        if (!done) {  // a partial never came: leave the slots, report
          if (lane == 0) atomicOr(p.err, PKV_ERR_TIMEOUT);
          return;
        }
        store_output<G>(out_row0, all, g8, tig);
        for (int gg = g_first; gg < g_last; ++gg) {
          float* q = p.slots + static_cast<size_t>(2 * gg + (gg == g_first ? 1 : 0)) * C::kSlotFloats;
          for (int i = lane; i < C::kSlotFloats; i += 32) q[i] = 0.f;
        }
      };
      // The segment continued from the previous group (its pieces open warp 0's
      // range and maybe the next ones) is merged by the last warp with no
      // segment of its own to merge, so that no warp merges two.
      const int first_bh0 = s_first_bh[0];
      int b_warp = 0;
      for (int w2 = kW - 1; w2 > 0; --w2)
        if (!s_has_head[w2]) {
          b_warp = w2;
          break;
        }
      if (first_bh0 >= 0 && warp == b_warp) {
        Piece pc;
        pc.m = -INFINITY;
        pc.l = 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d) pc.acc[d] = make_float2(0.f, 0.f);
        fold_run<G>(pc, s_slots, C::kSlotFloats, 1, g8, tig);
        const int2 gg = s_cont_groups;
        merge_segment(first_bh0, pc, 0, gg.x, gg.y);
      }
      const int3 head = s_head[warp];
      if (head.x >= 0) {  // this range's last piece, still in registers
        Piece pc;
#pragma unroll
        for (int d = 0; d < 8; ++d) pc.acc[d] = make_float2(o[d][0] + o[d][2], o[d][1] + o[d][3]);
        pc.l = l_run + __shfl_xor_sync(kFull, l_run, 1);
        pc.l += __shfl_xor_sync(kFull, pc.l, 2);
        pc.m = m_run;
        merge_segment(head.x, pc, warp, head.y, head.z);
      }
      __syncthreads();  // the slots are free for the next group
    }
  }

  if (failed) {
    // Report, then let every copy this warp may still have in flight land
    // before the CTA's shared memory is released.
    if (lane == 0) atomicOr(p.err, PKV_ERR_TIMEOUT);
    for (int s = 0; s < C::kStages; ++s) {
      const int st = (stage + s) % C::kStages;
      mbar_wait_bounded(bar0 + 8 * st, (phase_bits >> st) & 1u);
    }
  }
}


// One CTA: a step's plan (see kPlanHdr) for a decode launch of nwarps warps:
// every length checked as the decode checks it, the page prefix sums, the
// partition and the first item of every range.
constexpr int kPlanThreads = 1024;
__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ positions,
                int rope_positions, int batch, int hkv, int cap, int nwarps, int key,
                int* __restrict__ plan) {
  __shared__ int s_len[kDecodeBatchChunk], s_pre[kDecodeBatchChunk + 1], s_warp[kPlanThreads / 32];
  for (int b = threadIdx.x; b < batch; b += kPlanThreads) {
    int bad;
    s_len[b] = checked_length(seq_lens[b], cap, positions, b, rope_positions, &bad);
  }
  __syncthreads();
  scan_pages<kPlanThreads>(s_len, s_pre, batch, s_warp);
  const Partition pt = make_partition(s_pre[batch], batch, hkv, nwarps, 0);
  int* len = plan + kPlanHdr;
  int* pre = len + batch;
  int* bnd = pre + batch + 1;
  for (int b = threadIdx.x; b <= batch; b += kPlanThreads) {
    if (b < batch) len[b] = s_len[b];
    pre[b] = s_pre[b];
  }
  for (int r = threadIdx.x; r <= pt.n_ranges; r += kPlanThreads)
    bnd[r] = partition_item_at(pt, r * pt.cw, s_pre, batch, hkv);
  if (threadIdx.x == 0) {
    const int hdr[8] = {key, batch, pt.n_items, pt.pu, pt.su, pt.total_units, pt.cw, pt.n_ranges};
    for (int i = 0; i < 8; ++i) plan[i] = hdr[i];
  }
}

template <int G>
struct Launcher {
  using Fn = void (*)(CUtensorMap, DecodeParams);
  static Fn kernel(int mode) {
    return mode == kModePartials ? gqa_decode_kernel<G, kModePartials>
           : mode == kModeStep   ? gqa_decode_kernel<G, kModeStep>
                                 : gqa_decode_kernel<G, kModeDecode>;
  }

  static int blocks_per_sm(int device, int mode) {
    static std::atomic<int> cache[3][64];
    const int d = device & 63;
    int v = cache[mode][d].load(std::memory_order_relaxed);
    if (v > 0) return v;
    const size_t smem = smem_bytes<G>();
    if (cudaFuncSetAttribute(kernel(mode), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return -1;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel(mode), Cfg<G>::kThreads, smem) !=
        cudaSuccess)
      return -1;
    v = nb < 1 ? 1 : nb;
    cache[mode][d].store(v, std::memory_order_relaxed);
    return v;
  }

  // Launched with programmatic stream serialization: the kernel may start
  // while its predecessor in the stream finishes (see the kernel for what it
  // does before its dependency wait).
  static cudaError_t launch(const CUtensorMap& map, const DecodeParams& p, int grid,
                            cudaStream_t stream, int mode) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Cfg<G>::kThreads);
    cfg.dynamicSmemBytes = smem_bytes<G>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel(mode), map, p);
  }
};

#define PKV_FOR_GROUP(group, CALL)       \
  switch (group) {                       \
    case 1: return Launcher<1>::CALL;    \
    case 2: return Launcher<2>::CALL;    \
    case 3: return Launcher<3>::CALL;    \
    case 4: return Launcher<4>::CALL;    \
    case 5: return Launcher<5>::CALL;    \
    case 6: return Launcher<6>::CALL;    \
    case 7: return Launcher<7>::CALL;    \
    case 8: return Launcher<8>::CALL;    \
    default: break;                      \
  }

int blocks_per_sm_for(int group, int device, int mode) {
  PKV_FOR_GROUP(group, blocks_per_sm(device, mode));
  return -1;
}

cudaError_t launch_group(int group, const CUtensorMap& map, const DecodeParams& p, int grid,
                         cudaStream_t stream, int mode) {
  PKV_FOR_GROUP(group, launch(map, p, grid, stream, mode));
  return cudaErrorInvalidValue;
}

int warps_per_cta(int group) { return group <= 4 ? Cfg<4>::kWarps : Cfg<8>::kWarps; }

int slot_floats_for(int group) { return ((group * kHeadDim + 2 * group) + 3) / 4 * 4; }

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// The decode's grid: one CTA per SM (blocks_per_sm of them), less a few SMs
// (see launch_decode). 0 when the kernel cannot be configured.
int decode_grid(int group, int device, int mode) {
  const int bps = blocks_per_sm_for(group, device, mode);
  const int sms = device_sm_count(device);
  if (bps < 1 || sms < 1) return 0;
  return sms * bps > kSpareSms ? sms * bps - kSpareSms : sms * bps;
}

// Workspace layout for the automatic partition: the partial slots (two per
// warp of the grid), then the plan area.
size_t slots_bytes(int group, long long warps) {
  return static_cast<size_t>(2 * warps) * slot_floats_for(group) * sizeof(float);
}
size_t plan_bytes(int batch, long long warps) {
  return align256(sizeof(int) * (kPlanHdr + 2 * static_cast<size_t>(batch) + 1 +
                                 static_cast<size_t>(warps) + 1));
}

// The launch shape a plan is made for (never 0): kv heads, group, grid,
// warps per CTA, the length cap, and the RoPE table rows the lengths were
// checked against (0: positions not checked).
int plan_key(int hkv, int group, int grid, int cap, int rope_positions) {
  uint32_t h = 0x9e3779b9u;
  const uint32_t v[6] = {static_cast<uint32_t>(hkv), static_cast<uint32_t>(group),
                         static_cast<uint32_t>(grid), static_cast<uint32_t>(warps_per_cta(group)),
                         static_cast<uint32_t>(cap), static_cast<uint32_t>(rope_positions)};
  for (uint32_t x : v) h ^= x + 0x9e3779b9u + (h << 6) + (h >> 2);
  return static_cast<int>(h | 1u);
}

}  // namespace

size_t decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int max_blocks,
                              int pages_per_split, int sm_count) {
  if (batch < 0 || num_kv_heads < 1 || num_q_heads % num_kv_heads || max_blocks < 1 ||
      pages_per_split < 0 || sm_count < 1)
    return 0;
  const int group = num_q_heads / num_kv_heads;
  if (group < 1 || group > PKV_MAX_GROUP) return 0;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return 0;
  const int bps = blocks_per_sm_for(group, device, kModeDecode);
  if (bps < 1) return 0;
  const long long warps = static_cast<long long>(sm_count) * bps * warps_per_cta(group);
  long long ranges = warps;
  if (pages_per_split > 0) {
    const long long chunk = batch < kDecodeBatchChunk ? batch : kDecodeBatchChunk;
    const long long items = chunk * num_kv_heads * max_blocks;
    const long long need = (items + pages_per_split - 1) / pages_per_split;
    if (need > ranges) ranges = need;
    // two partial slots per group of ranges (a group has one range per warp of a CTA)
    return slots_bytes(group, ranges);
  }
  // the automatic partition: the slots, then (one launch) the step's plan
  size_t bytes = slots_bytes(group, warps);
  if (batch <= kDecodeBatchChunk) bytes = align256(bytes) + plan_bytes(batch, warps);
  return bytes;
}

cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* positions, int rope_positions,
                        int batch, int num_q_heads, int num_kv_heads, int max_blocks,
                        void* workspace, cudaStream_t stream) {
  if (batch == 0 || batch > kDecodeBatchChunk) return cudaSuccess;  // only one-launch batches
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const int group = num_q_heads / num_kv_heads;
  const int mode = positions ? kModeStep : kModeDecode;
  const int grid = decode_grid(group, device, mode);
  if (grid < 1) return cudaErrorInvalidConfiguration;
  const int cap = max_blocks * kPage;
  const int rp = positions ? rope_positions : 0;
  const int sms = device_sm_count(device);
  const long long warps = static_cast<long long>(sms) * blocks_per_sm_for(group, device, mode) *
                          warps_per_cta(group);
  int* plan = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) +
                                     align256(slots_bytes(group, warps)));
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(seq_lens, positions, rp, batch, num_kv_heads, cap,
                                              grid * warps_per_cta(group),
                                              plan_key(num_kv_heads, group, grid, cap, rp), plan);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const int group = a.num_q_heads / a.num_kv_heads;
  const bool partials = a.o_part != nullptr;
  const bool step = a.q_raw != nullptr;
  const int mode = partials ? kModePartials : step ? kModeStep : kModeDecode;
  const int bps = blocks_per_sm_for(group, device, mode);
  if (bps < 1) return cudaErrorInvalidConfiguration;
  const int sms = device_sm_count(device);
  if (sms < 1) return cudaErrorInvalidDevice;
  // A few SMs get no decode CTA: CTAs are placed in block order as the
  // previous kernel's CTAs leave their SMs, so the last ones would start
  // late (their set-up runs while the memory system is busiest) and finish
  // last; the page stream does not need every SM.
  const int grid = decode_grid(group, device, mode);
  // the step's plan, for the automatic partition of a one-launch batch
  const long long warps = static_cast<long long>(sms) * bps * warps_per_cta(group);
  const bool use_plan = !partials && a.pages_per_split == 0 && a.batch <= kDecodeBatchChunk &&
                        a.workspace != nullptr;
  const int* plan = use_plan ? reinterpret_cast<const int*>(static_cast<const uint8_t*>(a.workspace) +
                                                            align256(slots_bytes(group, warps)))
                             : nullptr;
  const int key = plan_key(a.num_kv_heads, group, grid, a.max_blocks * kPage,
                           step ? a.rope_positions : 0);
  const double log2e = 1.4426950408889634;
  for (int b0 = 0; b0 < a.batch; b0 += kDecodeBatchChunk) {
    const int nb = a.batch - b0 < kDecodeBatchChunk ? a.batch - b0 : kDecodeBatchChunk;
    DecodeParams p;
    p.num_pages = a.num_pages;
    p.hkv = a.num_kv_heads;
    p.q_rot = a.q_rot ? a.q_rot + static_cast<size_t>(b0) * a.num_q_heads * kHeadDim : nullptr;
    p.out = partials ? nullptr : a.out + static_cast<size_t>(b0) * a.num_q_heads * kHeadDim;
    p.block_tables = a.block_tables + static_cast<size_t>(b0) * a.max_blocks;
    p.max_blocks = a.max_blocks;
    p.seq_lens = a.seq_lens + b0;
    p.batch = nb;
    p.hq = a.num_q_heads;
    p.qscale = static_cast<float>(static_cast<double>(a.scale) * log2e);
    p.pages_per_split = a.pages_per_split;
    p.slots = partials ? nullptr : static_cast<float*>(a.workspace);
    const size_t row0 = static_cast<size_t>(b0) * a.num_q_heads;
    p.o_part = partials ? a.o_part + row0 * a.max_splits * kHeadDim : nullptr;
    p.lse_part = partials ? a.lse_part + row0 * a.max_splits : nullptr;
    p.num_splits = partials ? a.num_splits + row0 : nullptr;
    p.max_splits = a.max_splits;
    p.err = a.err;
    p.merge_looks = a.merge_looks;
    p.plan = plan;
    p.plan_key = key;
    p.ring_offset = static_cast<int>(ring_offset_bytes());
    const size_t qrow0 = static_cast<size_t>(b0) * a.num_q_heads * kHeadDim;
    const size_t krow0 = static_cast<size_t>(b0) * a.num_kv_heads * kHeadDim;
    p.q_raw = step ? a.q_raw + qrow0 : nullptr;
    p.k_new = step ? a.k_new + krow0 : nullptr;
    p.v_new = step ? a.v_new + krow0 : nullptr;
    // the fp32 pair rows, then the fp64 rows (see launch_rope_cos_sin), one
    // row per position
    p.rope_ff = step ? static_cast<const float4*>(a.rope_table) : nullptr;
    p.rope_dd = step ? reinterpret_cast<const double2*>(static_cast<const float4*>(a.rope_table) +
                                                        static_cast<size_t>(a.rope_positions) * kHalfDim)
                     : nullptr;
    p.positions = step ? a.positions + b0 : nullptr;
    p.rope_positions = a.rope_positions;
    p.q_rot_out = (step && a.q_rot_out) ? a.q_rot_out + qrow0 : nullptr;
    p.pool_w = const_cast<uint8_t*>(a.pool);
    e = launch_group(group, *a.kv_map, p, grid, stream, mode);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pkv
