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
// Design (GB300-first, HBM bound: per token and kv head it reads 256 B and
// does 256*G flops, G = 4 or 7 on the two model shapes):
//  * Work items are (sequence, kv head, page) triples, enumerated sequence-
//    major. A persistent grid of one CTA per SM (8 warps) cuts the item list
//    into equal contiguous ranges, one range per warp, so long and short
//    sequences balance at page granularity with no host-side planning.
//  * Each warp streams its range through its own 4-stage shared-memory ring:
//    lane 0 issues 1-D bulk asynchronous copies (cp.async.bulk, completion
//    counted in bytes on an mbarrier) of the head's 2 KiB K block and 2 KiB V
//    block of each page, only the valid rows of a partial last page, plus the
//    G query rows whenever a new (sequence, head) piece starts. No thread
//    spends registers or issue slots on global loads.
//  * In a warp, lane (t, c) = (lane>>3, lane&7) holds dims [8c, 8c+8) of token
//    row t of a 4-row step; q for those dims and all G heads stays in
//    registers. Partial dot products are reduced over the 8 lanes of a row
//    with an exchanging butterfly that leaves each lane one head's score, so
//    each score is exponentiated once. Softmax state is per page: one max
//    per head over the page's 16 tokens, one rescale of the accumulators when
//    the max grows. Products use the packed fp32x2 FMA of sm_100+.
//  * A (sequence, head) piece that spans several warp ranges writes its
//    unnormalised accumulator, max and sum to a workspace slot; the last warp
//    to arrive (an atomic counter per (sequence, head)) merges the pieces and
//    resets the counter. Nothing ever waits on another warp.
#include <atomic>
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr int kHdrBytes = 512;  // mbarriers (kWarps*kStages*8 = 256 B) + scan scratch
constexpr int kScanScratch = 256;
constexpr int kStepBytes = 4 * kRowBytes;  // 4 token rows per warp step = 512 B
constexpr float kLn2 = 0.6931471805599453f;

template <int G>
struct Geo {
  static constexpr int GP = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;  // padded to a power of 2
  static constexpr int kLogGP = GP == 1 ? 0 : GP == 2 ? 1 : GP == 4 ? 2 : 3;
  static constexpr int kShift = 3 - kLogGP;  // head of lane = (lane & 7) >> kShift
  static constexpr int kQBytes = G * kHeadDim * 4;
  static constexpr int kStageBytes = kHeadPageBytes + ((kQBytes + 127) / 128) * 128;
  static constexpr int kSlotFloats = ((G * kHeadDim + 2 * G) + 3) / 4 * 4;
};

struct DecodeParams {
  const uint8_t* pool;
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
  int* counters;  // [batch][hkv]
  float* slots;
  float* o_part;
  float* lse_part;
  int32_t* num_splits;
  int max_splits;
  int* err;
  int ring_offset;  // byte offset of the copy rings in dynamic shared memory
};

size_t ring_offset_bytes() {
  return static_cast<size_t>(kHdrBytes) +
         ((sizeof(int) * (2 * kDecodeBatchChunk + 1) + 127) / 128) * 128;
}

template <int G>
size_t smem_bytes() {
  return ring_offset_bytes() + static_cast<size_t>(kWarps) * kStages * Geo<G>::kStageBytes;
}

// Butterfly over the 8 lanes of a token row that halves the number of values
// each lane carries at every level it can: on return v[0] is, for head
// (lane & 7) >> (3 - log2 GP), the sum of the 8 lanes' partial dot products.
template <int GP>
__device__ __forceinline__ float exchange_reduce(float (&v)[GP], int lane) {
#pragma unroll
  for (int level = 0; level < 3; ++level) {
    const int mask = 4 >> level;
    const int n = GP >> level;
    if (n >= 2) {
      const bool upper = (lane & mask) != 0;
#pragma unroll
      for (int j = 0; j < n / 2; ++j) {
        const float send = upper ? v[j] : v[j + n / 2];
        const float keep = upper ? v[j + n / 2] : v[j];
        v[j] = keep + __shfl_xor_sync(kFull, send, mask);
      }
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], mask);
    }
  }
  return v[0];
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

__device__ __forceinline__ void advance(Cursor& c, const int* s_pre, const int* s_len, int batch,
                                        int hkv) {
  ++c.item;
  if (++c.pg < c.np) return;
  c.pg = 0;
  if (++c.h < hkv) return;
  c.h = 0;
  do {
    ++c.b;
  } while (c.b < batch && s_len[c.b] == 0);
  if (c.b < batch) {
    c.np = s_pre[c.b + 1] - s_pre[c.b];
    c.len = s_len[c.b];
  }
}

// Exclusive prefix sum of pages per sequence into s_pre[0..batch], total last.
__device__ void scan_pages(const int* s_len, int* s_pre, int batch, int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (batch + kThreads - 1) / kThreads;
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
  int wofs = 0;
  for (int w = 0; w < warp; ++w) wofs += s_warp[w];
  int run = wofs + incl - local;
  for (int b = beg; b < end; ++b) {
    s_pre[b] = run;
    run += (s_len[b] + kPage - 1) / kPage;
  }
  if (tid == kThreads - 1) s_pre[batch] = wofs + incl;
  __syncthreads();
}

template <int G, bool kPartials>
__global__ void __launch_bounds__(kThreads, 1) gqa_decode_kernel(const DecodeParams p) {
  using Ge = Geo<G>;
  constexpr int GP = Ge::GP;
  constexpr int kShift = Ge::kShift;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tg = lane >> 3;         // token row within a 4-row step
  const int c8 = (lane & 7) * 8;    // first of this lane's 8 dims
  int* s_warp = reinterpret_cast<int*>(smem + kHdrBytes - kScanScratch);
  int* s_len = reinterpret_cast<int*>(smem + kHdrBytes);
  int* s_pre = s_len + p.batch;
  __shared__ int s_bad_len;
  const uint32_t bar0 = smem_addr(smem) + warp * kStages * 8;
  const uint32_t ring0 = smem_addr(smem + p.ring_offset) + warp * kStages * Ge::kStageBytes;

  // Sequence lengths (invalid ones become empty) and the page prefix sums.
  if (tid == 0) s_bad_len = 0;
  if (lane == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
  fence_mbar_init();
  __syncthreads();
  const int cap = p.max_blocks * kPage;
  for (int b = tid; b < p.batch; b += kThreads) {
    int n = p.seq_lens[b];
    if (n < 1 || n > cap) {
      n = 0;
      s_bad_len = 1;
    }
    s_len[b] = n;
  }
  __syncthreads();
  scan_pages(s_len, s_pre, p.batch, s_warp);

  if (s_bad_len) {  // rows of invalid sequences: zero output (or zero split count)
    if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, PKV_ERR_SEQ_LEN);
    const int rows = p.batch * p.hq;
    for (int idx = blockIdx.x * kThreads + tid; idx < rows; idx += gridDim.x * kThreads) {
      if (s_len[idx / p.hq] != 0) continue;
      if (kPartials) {
        p.num_splits[idx] = 0;
      } else {
        float4* o = reinterpret_cast<float4*>(p.out + static_cast<size_t>(idx) * kHeadDim);
#pragma unroll
        for (int k = 0; k < kHeadDim / 4; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  const int n_items = s_pre[p.batch] * p.hkv;
  if (n_items == 0) return;
  const int nwarps = gridDim.x * kWarps;
  const int c = p.pages_per_split > 0 ? p.pages_per_split : (n_items + nwarps - 1) / nwarps;
  const int n_ranges = (n_items + c - 1) / c;
  const float qs = p.qscale;

  uint32_t phase_bits = 0;  // bit s: parity of the next completion of stage s
  int stage = 0;            // next stage to consume
  uint32_t bad_bits = 0;    // bit s: stage s carries no K/V (bad page id)
  bool failed = false;
  int win_b = -1, win_base = 0, win_val = -1;  // lane-parallel window of one block-table row

  auto issue = [&](const Cursor& pc, bool first, int st) {
    if (pc.b != win_b || pc.pg < win_base || pc.pg >= win_base + 32) {
      win_b = pc.b;
      win_base = pc.pg & ~31;
      const int idx = win_base + lane;
      win_val = idx < p.max_blocks
                    ? __ldg(p.block_tables + static_cast<size_t>(pc.b) * p.max_blocks + idx)
                    : -1;
    }
    const int page = __shfl_sync(kFull, win_val, pc.pg - win_base);
    const bool bad = page < 0 || static_cast<long long>(page) >= p.num_pages;
    const int nv = min(kPage, pc.len - pc.pg * kPage);
    bad_bits = bad ? (bad_bits | (1u << st)) : (bad_bits & ~(1u << st));
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t dst = ring0 + st * Ge::kStageBytes;
      const uint32_t bytes = (bad ? 0u : 2u * nv * kRowBytes) + (first ? Ge::kQBytes : 0u);
      if (bad) atomicOr(p.err, PKV_ERR_PAGE_ID);
      if (bytes == 0) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, bytes);
        if (!bad) {
          const uint8_t* src =
              p.pool + (static_cast<size_t>(page) * p.hkv + pc.h) * kHeadPageBytes;
          bulk_g2s(dst, src, nv * kRowBytes, bar);
          bulk_g2s(dst + kHalfBytes, src + kHalfBytes, nv * kRowBytes, bar);
        }
        if (first)
          bulk_g2s(dst + kHeadPageBytes,
                   p.q_rot + (static_cast<size_t>(pc.b) * p.hq + pc.h * G) * kHeadDim,
                   Ge::kQBytes, bar);
      }
    }
  };

  float2 q2[G][4];
  float2 acc[G][4];
  float m_own = -INFINITY, l_own = 0.f;

  for (int r = blockIdx.x * kWarps + warp; r < n_ranges && !failed; r += nwarps) {
    const int i0 = r * c, i1 = min(i0 + c, n_items);
    Cursor cur = locate(i0, s_pre, s_len, p.batch, p.hkv);
    Cursor pc = cur;
    {
      int st = stage;
      for (int k = 0; k < kStages && i0 + k < i1; ++k) {
        issue(pc, pc.item == i0 || pc.pg == 0, st);
        advance(pc, s_pre, s_len, p.batch, p.hkv);
        st = (st + 1 == kStages) ? 0 : st + 1;
      }
    }
    int start_pg = 0;
    bool first_in_range = true;
    for (int i = i0; i < i1; ++i) {
      const int st = stage;
      if (!mbar_wait_bounded(bar0 + 8 * st, (phase_bits >> st) & 1u)) {
        failed = true;
        break;
      }
      phase_bits ^= 1u << st;
      const uint32_t sbase = ring0 + st * Ge::kStageBytes;
      const bool first = (i == i0) || cur.pg == 0;
      const bool last = (i == i1 - 1) || cur.pg == cur.np - 1;
      if (first) {
        start_pg = cur.pg;
        first_in_range = (i == i0);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 a = lds128f(sbase + kHeadPageBytes + (g * kHeadDim + c8) * 4);
          const float4 e = lds128f(sbase + kHeadPageBytes + (g * kHeadDim + c8 + 4) * 4);
          q2[g][0] = make_float2(a.x * qs, a.y * qs);
          q2[g][1] = make_float2(a.z * qs, a.w * qs);
          q2[g][2] = make_float2(e.x * qs, e.y * qs);
          q2[g][3] = make_float2(e.z * qs, e.w * qs);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[g][j] = make_float2(0.f, 0.f);
        }
        m_own = -INFINITY;
        l_own = 0.f;
      }
      if (!((bad_bits >> st) & 1u)) {
        const int nv = min(kPage, cur.len - cur.pg * kPage);
        // Scores of the page's 16 tokens: this lane ends with token 4r+tg, head (lane&7)>>kShift.
        float s[4];
#pragma unroll
        for (int rs = 0; rs < 4; ++rs) {
          const uint4 kw = lds128(sbase + rs * kStepBytes + lane * 16);
          const float2 k0 = bf16x2_to_float2(kw.x), k1 = bf16x2_to_float2(kw.y);
          const float2 k2 = bf16x2_to_float2(kw.z), k3 = bf16x2_to_float2(kw.w);
          float part[GP];
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            if (g < G) {
              float2 t = __fmul2_rn(q2[g][0], k0);
              t = __ffma2_rn(q2[g][1], k1, t);
              t = __ffma2_rn(q2[g][2], k2, t);
              t = __ffma2_rn(q2[g][3], k3, t);
              part[g] = t.x + t.y;
            } else {
              part[g] = 0.f;
            }
          }
          s[rs] = exchange_reduce<GP>(part, lane);
        }
        if (nv < kPage) {
#pragma unroll
          for (int rs = 0; rs < 4; ++rs)
            if (rs * 4 + tg >= nv) s[rs] = -INFINITY;
        }
        float pm = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
        pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 8));
        pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 16));
        const float m_new = fmaxf(m_own, pm);
        const bool grew = m_new > m_own;
        const float alpha = grew ? fast_exp2(m_own - m_new) : 1.f;
        float pr[4];
#pragma unroll
        for (int rs = 0; rs < 4; ++rs) pr[rs] = fast_exp2(s[rs] - m_new);
        l_own = l_own * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
        m_own = m_new;
        if (__any_sync(kFull, grew)) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float a = __shfl_sync(kFull, alpha, (lane & ~7) | (g << kShift));
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[g][j] = __fmul2_rn(acc[g][j], a2);
          }
        }
#pragma unroll
        for (int rs = 0; rs < 4; ++rs) {
          const uint4 vw = lds128(sbase + kHalfBytes + rs * kStepBytes + lane * 16);
          float2 v0 = bf16x2_to_float2(vw.x), v1 = bf16x2_to_float2(vw.y);
          float2 v2 = bf16x2_to_float2(vw.z), v3 = bf16x2_to_float2(vw.w);
          if (nv < kPage && rs * 4 + tg >= nv) {  // stale shared memory past the valid rows
            v0 = v1 = v2 = v3 = make_float2(0.f, 0.f);
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pg = __shfl_sync(kFull, pr[rs], (lane & ~7) | (g << kShift));
            const float2 p2 = make_float2(pg, pg);
            acc[g][0] = __ffma2_rn(p2, v0, acc[g][0]);
            acc[g][1] = __ffma2_rn(p2, v1, acc[g][1]);
            acc[g][2] = __ffma2_rn(p2, v2, acc[g][2]);
            acc[g][3] = __ffma2_rn(p2, v3, acc[g][3]);
          }
        }
      }

      if (last) {
        // Sum the four token rows' accumulators and sums; fetch each head's max and sum.
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[g][j].x += __shfl_xor_sync(kFull, acc[g][j].x, 8);
            acc[g][j].y += __shfl_xor_sync(kFull, acc[g][j].y, 8);
            acc[g][j].x += __shfl_xor_sync(kFull, acc[g][j].x, 16);
            acc[g][j].y += __shfl_xor_sync(kFull, acc[g][j].y, 16);
          }
        l_own += __shfl_xor_sync(kFull, l_own, 8);
        l_own += __shfl_xor_sync(kFull, l_own, 16);
        float mh[G], lh[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          mh[g] = __shfl_sync(kFull, m_own, g << kShift);
          lh[g] = __shfl_sync(kFull, l_own, g << kShift);
        }
        const int seg_start = p.hkv * s_pre[cur.b] + cur.h * cur.np;
        const int pieces = (seg_start + cur.np - 1) / c - seg_start / c + 1;
        const size_t row0 = static_cast<size_t>(cur.b) * p.hq + cur.h * G;
        const bool complete = (start_pg == 0) && (cur.pg == cur.np - 1);
        if (kPartials) {
          const int j = r - seg_start / c;
          if (pieces > p.max_splits) {
            if (lane == 0) atomicOr(p.err, PKV_ERR_SPLITS);
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const size_t row = row0 + g;
              if ((g & 3) == tg) {
                const float inv = lh[g] > 0.f ? 1.f / lh[g] : 0.f;
                float4* o = reinterpret_cast<float4*>(
                    p.o_part + (row * p.max_splits + j) * kHeadDim + c8);
                o[0] = make_float4(acc[g][0].x * inv, acc[g][0].y * inv, acc[g][1].x * inv,
                                   acc[g][1].y * inv);
                o[1] = make_float4(acc[g][2].x * inv, acc[g][2].y * inv, acc[g][3].x * inv,
                                   acc[g][3].y * inv);
              }
              if (lane == g) {
                p.lse_part[row * p.max_splits + j] =
                    lh[g] > 0.f ? (mh[g] + __log2f(lh[g])) * kLn2 : -INFINITY;
                p.num_splits[row] = pieces;
              }
            }
          }
        } else if (complete) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            if ((g & 3) == tg) {
              const float inv = lh[g] > 0.f ? 1.f / lh[g] : 0.f;
              float4* o = reinterpret_cast<float4*>(p.out + (row0 + g) * kHeadDim + c8);
              o[0] = make_float4(acc[g][0].x * inv, acc[g][0].y * inv, acc[g][1].x * inv,
                                 acc[g][1].y * inv);
              o[1] = make_float4(acc[g][2].x * inv, acc[g][2].y * inv, acc[g][3].x * inv,
                                 acc[g][3].y * inv);
            }
          }
        } else {
          // A piece of a split (sequence, head): publish it, and merge if last.
          float* sp = p.slots + static_cast<size_t>(2 * r + (first_in_range ? 0 : 1)) *
                                    Ge::kSlotFloats;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            if ((g & 3) == tg) {
              float4* o = reinterpret_cast<float4*>(sp + g * kHeadDim + c8);
              o[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
              o[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
            }
            if (lane == g) {
              sp[G * kHeadDim + g] = mh[g];
              sp[G * kHeadDim + G + g] = lh[g];
            }
          }
          __threadfence();
          __syncwarp();
          int old = 0;
          int* counter = p.counters + cur.b * p.hkv + cur.h;
          if (lane == 0) old = atomicAdd(counter, 1);
          old = __shfl_sync(kFull, old, 0);
          if (old == pieces - 1) {
            __threadfence();
            const int r0 = seg_start / c;
            const bool r0_mid = (seg_start != r0 * c);  // piece 0 is range r0's last segment
#pragma unroll 1
            for (int g = 0; g < G; ++g) {
              float mx = -INFINITY;
              for (int jp = 0; jp < pieces; ++jp) {
                const int slot = 2 * (r0 + jp) + ((jp == 0 && r0_mid) ? 1 : 0);
                mx = fmaxf(mx, ld_cg(p.slots + static_cast<size_t>(slot) * Ge::kSlotFloats +
                                     G * kHeadDim + g));
              }
              float lsum = 0.f;
              float2 o = make_float2(0.f, 0.f);
              for (int jp = 0; jp < pieces; ++jp) {
                const int slot = 2 * (r0 + jp) + ((jp == 0 && r0_mid) ? 1 : 0);
                const float* q = p.slots + static_cast<size_t>(slot) * Ge::kSlotFloats;
                const float mj = ld_cg(q + G * kHeadDim + g);
                const float w = (mj == -INFINITY) ? 0.f : fast_exp2(mj - mx);
                lsum += w * ld_cg(q + G * kHeadDim + G + g);
                const float2 a = ld_cg2(reinterpret_cast<const float2*>(q + g * kHeadDim) + lane);
                o.x += w * a.x;
                o.y += w * a.y;
              }
              const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
              reinterpret_cast<float2*>(p.out + (row0 + g) * kHeadDim)[lane] =
                  make_float2(o.x * inv, o.y * inv);
            }
            if (lane == 0) *counter = 0;
          }
        }
      }

      fence_proxy_async_smem();
      __syncwarp();
      if (i + kStages < i1) {
        issue(pc, pc.pg == 0, st);
        advance(pc, s_pre, s_len, p.batch, p.hkv);
      }
      advance(cur, s_pre, s_len, p.batch, p.hkv);
      stage = (stage + 1 == kStages) ? 0 : stage + 1;
    }
  }

  if (failed) {
    // Report, then let every copy this warp may still have in flight land
    // before the CTA's shared memory is released.
    if (lane == 0) atomicOr(p.err, PKV_ERR_TIMEOUT);
    for (int s = 0; s < kStages; ++s) {
      const int st = (stage + s) % kStages;
      mbar_wait_bounded(bar0 + 8 * st, (phase_bits >> st) & 1u);
    }
  }
}

template <int G>
struct Occupancy {
  static int blocks_per_sm(int device, bool partials) {
    static std::atomic<int> cache[2][64];
    const int d = device & 63;
    int v = cache[partials][d].load(std::memory_order_relaxed);
    if (v > 0) return v;
    const size_t smem = smem_bytes<G>();
    auto fn_f = gqa_decode_kernel<G, false>;
    auto fn_p = gqa_decode_kernel<G, true>;
    if (cudaFuncSetAttribute(fn_f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(fn_p, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return -1;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, partials ? fn_p : fn_f, kThreads, smem) !=
        cudaSuccess)
      return -1;
    v = nb < 1 ? 1 : nb;
    cache[partials][d].store(v, std::memory_order_relaxed);
    return v;
  }
};

int blocks_per_sm_for(int group, int device, bool partials) {
  switch (group) {
    case 1: return Occupancy<1>::blocks_per_sm(device, partials);
    case 2: return Occupancy<2>::blocks_per_sm(device, partials);
    case 3: return Occupancy<3>::blocks_per_sm(device, partials);
    case 4: return Occupancy<4>::blocks_per_sm(device, partials);
    case 5: return Occupancy<5>::blocks_per_sm(device, partials);
    case 6: return Occupancy<6>::blocks_per_sm(device, partials);
    case 7: return Occupancy<7>::blocks_per_sm(device, partials);
    case 8: return Occupancy<8>::blocks_per_sm(device, partials);
    default: return -1;
  }
}

int slot_floats_for(int group) {
  return ((group * kHeadDim + 2 * group) + 3) / 4 * 4;
}

template <int G>
cudaError_t launch_g(const DecodeParams& p, int grid, cudaStream_t stream, bool partials) {
  const size_t smem = smem_bytes<G>();
  if (partials)
    gqa_decode_kernel<G, true><<<grid, kThreads, smem, stream>>>(p);
  else
    gqa_decode_kernel<G, false><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
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
  const int bps = blocks_per_sm_for(group, device, false);
  if (bps < 1) return 0;
  const long long warps = static_cast<long long>(sm_count) * bps * kWarps;
  long long ranges = warps;
  if (pages_per_split > 0) {
    const long long chunk = batch < kDecodeBatchChunk ? batch : kDecodeBatchChunk;
    const long long items = chunk * num_kv_heads * max_blocks;
    const long long need = (items + pages_per_split - 1) / pages_per_split;
    if (need > ranges) ranges = need;
  }
  const size_t counters = ((static_cast<size_t>(batch) * num_kv_heads * sizeof(int) + 255) / 256) * 256;
  const size_t slots = static_cast<size_t>(2 * ranges) * slot_floats_for(group) * sizeof(float);
  return counters + slots;
}

cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  const int group = a.num_q_heads / a.num_kv_heads;
  const bool partials = a.o_part != nullptr;
  const int bps = blocks_per_sm_for(group, device, partials);
  if (bps < 1) return cudaErrorInvalidConfiguration;
  const int sms = device_sm_count(device);
  if (sms < 1) return cudaErrorInvalidDevice;
  const int grid = sms * bps;
  const size_t counters_bytes =
      ((static_cast<size_t>(a.batch) * a.num_kv_heads * sizeof(int) + 255) / 256) * 256;
  const double log2e = 1.4426950408889634;
  for (int b0 = 0; b0 < a.batch; b0 += kDecodeBatchChunk) {
    const int nb = a.batch - b0 < kDecodeBatchChunk ? a.batch - b0 : kDecodeBatchChunk;
    DecodeParams p;
    p.pool = a.pool;
    p.num_pages = a.num_pages;
    p.hkv = a.num_kv_heads;
    p.q_rot = a.q_rot + static_cast<size_t>(b0) * a.num_q_heads * kHeadDim;
    p.out = partials ? nullptr : a.out + static_cast<size_t>(b0) * a.num_q_heads * kHeadDim;
    p.block_tables = a.block_tables + static_cast<size_t>(b0) * a.max_blocks;
    p.max_blocks = a.max_blocks;
    p.seq_lens = a.seq_lens + b0;
    p.batch = nb;
    p.hq = a.num_q_heads;
    p.qscale = static_cast<float>(static_cast<double>(a.scale) * log2e);
    p.pages_per_split = a.pages_per_split;
    p.counters = partials ? nullptr
                          : static_cast<int*>(a.workspace) + static_cast<size_t>(b0) * a.num_kv_heads;
    p.slots = partials ? nullptr
                       : reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + counters_bytes);
    const size_t row0 = static_cast<size_t>(b0) * a.num_q_heads;
    p.o_part = partials ? a.o_part + row0 * a.max_splits * kHeadDim : nullptr;
    p.lse_part = partials ? a.lse_part + row0 * a.max_splits : nullptr;
    p.num_splits = partials ? a.num_splits + row0 : nullptr;
    p.max_splits = a.max_splits;
    p.err = a.err;
    p.ring_offset = static_cast<int>(ring_offset_bytes());
    switch (group) {
      case 1: e = launch_g<1>(p, grid, stream, partials); break;
      case 2: e = launch_g<2>(p, grid, stream, partials); break;
      case 3: e = launch_g<3>(p, grid, stream, partials); break;
      case 4: e = launch_g<4>(p, grid, stream, partials); break;
      case 5: e = launch_g<5>(p, grid, stream, partials); break;
      case 6: e = launch_g<6>(p, grid, stream, partials); break;
      case 7: e = launch_g<7>(p, grid, stream, partials); break;
      case 8: e = launch_g<8>(p, grid, stream, partials); break;
      default: e = cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pkv
