// prefill.cu -- chunked causal prefill into the page pool.
//
// "Hours of YouTube and 85 handtyped pages of notes on LLM Inference – Start
// here": prefill fills the prompt pages (dense causal prefill), decode then
// appends one token at a time. A chunk of new tokens for sequence b sits at
// positions start_pos[b], start_pos[b]+1, ...; every chunk token is rotated
// and appended like a decode token, and the queries of chunk token t attend
// causally over the sequence's first start_pos[b] + t + 1 tokens.
//
// Three launches. (1) A preparation kernel: one block lists the query tiles,
// the others give every chunk token its sequence and position. (2) The append
// kernel rotates and stores every chunk token exactly as a decode token would
// be stored (cos and sin from the row of its position in the caller's RoPE
// table, built once for all positions), and writes the rotated queries.
// (3) Flash attention on the fifth-generation tensor
// cores: one CTA per (tile of up to 128 (token, query head) rows, kv head)
// streams the sequence's pages up to the tile's last position, four pages
// per step, through a TMA ring; tcgen05 MMAs with fp32 accumulators in tensor
// memory compute S = Q K^T and O += P V, and four threads per row (16 keys
// each) run the online softmax on its row of S.
#include <atomic>
#include <climits>
#include <cub/block/block_scan.cuh>

#include "pkv_device.cuh"
#include "tc05.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kHalfDim = kHeadDim / 2;

// One thread per chunk token: find its sequence by bisection over cu_tokens
// and write it and its position; a token of a malformed chunk (a decreasing
// cu_tokens, a negative start, or a position past max_blocks*16) gets
// sequence -PKV_ERR_SEQ_LEN, one at a position past the RoPE table's rows
// -PKV_ERR_POSITION, and position 0.
__device__ void expand_token(int idx, int max_blocks, int rope_positions,
                             const int32_t* __restrict__ cu_tokens,
                             const int32_t* __restrict__ start_pos, int batch, int total,
                             int32_t* __restrict__ tok_seq, int32_t* __restrict__ tok_pos) {
  if (idx >= total) return;
  int lo = 0, hi = batch - 1;  // largest b with cu_tokens[b] <= idx
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_tokens[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  const int c0 = cu_tokens[lo], c1 = cu_tokens[lo + 1];
  const long long pos = static_cast<long long>(start_pos[lo]) + (idx - c0);
  int why = 0;
  if (!(c0 <= idx && idx < c1 && start_pos[lo] >= 0 &&
        pos + 1 <= static_cast<long long>(max_blocks) * kPage))
    why = PKV_ERR_SEQ_LEN;
  else if (pos >= rope_positions)
    why = PKV_ERR_POSITION;
  tok_seq[idx] = why ? -why : lo;
  tok_pos[idx] = why ? 0 : static_cast<int32_t>(pos);
}

// One CTA per chunk token: its rotated query (fp32, from the fp32 cos/sin of
// the RoPE table row of its position), its key rotated and rounded to bf16
// exactly as fp64 arithmetic rounds it (the certified fp32 double-word path,
// fp64 from the table where it cannot certify: the bytes the decode append
// stores), and its value, both stored at its position in its sequence's
// pages. A token of a malformed chunk (position 0) still gets a rotated query.
// A thread loads its first two query items (four pairs each), its first two
// key pairs, its first 16-byte piece of the value rows and the block-table
// entry before the barrier that makes the cos/sin row visible, so that the
// token costs two dependent round trips (its position, then the rest) for
// the usual shapes (up to 64 query and 8 kv heads); items past those are
// loaded in the loops.
constexpr int kAppendThreads = 128;
__global__ void __launch_bounds__(kAppendThreads)
    prefill_append_kernel(uint16_t* __restrict__ pool, long long num_pages, int hkv, int hq,
                          const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                          const uint16_t* __restrict__ v, float* __restrict__ q_rot,
                          const int32_t* __restrict__ block_tables, int max_blocks,
                          const int32_t* __restrict__ tok_seq, const int32_t* __restrict__ tok_pos,
                          const float4* __restrict__ rope_ff, const double2* __restrict__ rope_dd,
                          int* __restrict__ err) {
  __shared__ float4 cs[kHalfDim];
  const int tkn = blockIdx.x, tid = threadIdx.x;
  const int b = tok_seq[tkn];
  const int pos = tok_pos[tkn];  // also the token's row of the RoPE table (0 when malformed)
  const int nq = hq * (kHalfDim / 4), nk = hkv * kHalfDim, nv = hkv * (kRowBytes / 16);
  const uint16_t* qb = q + static_cast<size_t>(tkn) * hq * kHeadDim;
  const uint16_t* kb = k + static_cast<size_t>(tkn) * hkv * kHeadDim;
  const uint4* vb = reinterpret_cast<const uint4*>(v + static_cast<size_t>(tkn) * hkv * kHeadDim);
  // query item idx: head idx / 8, pairs j0 .. j0 + 3 (8-byte loads of the
  // bf16 halves j0 .. j0 + 3 and j0 + 32 .. j0 + 35)
  auto q_load = [&](int idx, uint2& a, uint2& c) {
    const int head = idx / (kHalfDim / 4), j0 = 4 * (idx - head * (kHalfDim / 4));
    a = *reinterpret_cast<const uint2*>(qb + head * kHeadDim + j0);
    c = *reinterpret_cast<const uint2*>(qb + head * kHeadDim + j0 + kHalfDim);
  };
  auto k_load = [&](int idx, uint16_t& k0, uint16_t& k1) {
    const int hh = idx / kHalfDim, j = idx - hh * kHalfDim;
    k0 = kb[hh * kHeadDim + j];
    k1 = kb[hh * kHeadDim + j + kHalfDim];
  };
  uint2 qa0 = make_uint2(0u, 0u), qc0 = qa0, qa1 = qa0, qc1 = qa0;
  uint16_t k00 = 0, k10 = 0, k01 = 0, k11 = 0;
  uint4 v0 = make_uint4(0u, 0u, 0u, 0u);
  long long page = -1;
  if (tid < nq) q_load(tid, qa0, qc0);
  if (tid + kAppendThreads < nq) q_load(tid + kAppendThreads, qa1, qc1);
  if (b >= 0) {
    page = block_tables[static_cast<size_t>(b) * max_blocks + pos / kPage];
    if (tid < nk) k_load(tid, k00, k10);
    if (tid + kAppendThreads < nk) k_load(tid + kAppendThreads, k01, k11);
    if (tid < nv) v0 = vb[tid];
  }
  if (tid < kHalfDim) cs[tid] = rope_ff[static_cast<size_t>(pos) * kHalfDim + tid];
  __syncthreads();
  // the rotated query: 16-byte stores of the fp32 results
  float* qo = q_rot + static_cast<size_t>(tkn) * hq * kHeadDim;
  auto q_rotate = [&](int idx, uint2 a, uint2 c) {
    const int head = idx / (kHalfDim / 4), j0 = 4 * (idx - head * (kHalfDim / 4));
    const float x0[4] = {__uint_as_float(a.x << 16), __uint_as_float(a.x & 0xffff0000u),
                         __uint_as_float(a.y << 16), __uint_as_float(a.y & 0xffff0000u)};
    const float x1[4] = {__uint_as_float(c.x << 16), __uint_as_float(c.x & 0xffff0000u),
                         __uint_as_float(c.y << 16), __uint_as_float(c.y & 0xffff0000u)};
    float y0[4], y1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 t = cs[j0 + e];
      y0[e] = x0[e] * t.x - x1[e] * t.z;
      y1[e] = x1[e] * t.x + x0[e] * t.z;
    }
    *reinterpret_cast<float4*>(qo + head * kHeadDim + j0) = make_float4(y0[0], y0[1], y0[2], y0[3]);
    *reinterpret_cast<float4*>(qo + head * kHeadDim + j0 + kHalfDim) = make_float4(y1[0], y1[1], y1[2], y1[3]);
  };
  if (tid < nq) q_rotate(tid, qa0, qc0);
  if (tid + kAppendThreads < nq) q_rotate(tid + kAppendThreads, qa1, qc1);
  for (int idx = tid + 2 * kAppendThreads; idx < nq; idx += kAppendThreads) {
    uint2 a, c;
    q_load(idx, a, c);
    q_rotate(idx, a, c);
  }
  if (b < 0) {  // a malformed chunk, or a position past the RoPE table
    if (tid == 0) atomicOr(err, -b);
    return;
  }
  if (page < 0 || page >= num_pages) {
    if (tid == 0) atomicOr(err, PKV_ERR_PAGE_ID);
    return;
  }
  const int slot = pos % kPage;
  uint16_t* page_base = pool + static_cast<size_t>(page) * hkv * (kHeadPageBytes / 2);
  auto k_store = [&](int idx, uint16_t k0, uint16_t k1) {
    const int hh = idx / kHalfDim, j = idx - hh * kHalfDim;
    const float x0 = __uint_as_float(static_cast<uint32_t>(k0) << 16);
    const float x1 = __uint_as_float(static_cast<uint32_t>(k1) << 16);
    const float4 c = cs[j];
    uint16_t y0, y1;
    if (!(rotated_bf16_fast(x0, x1, c.x, c.y, c.z, c.w, y0) &&
          rotated_bf16_fast(x1, -x0, c.x, c.y, c.z, c.w, y1))) {
      const double2 cd = rope_dd[static_cast<size_t>(pos) * kHalfDim + j];
      rotate_key_pair(k0, k1, cd.x, cd.y, y0, y1);
    }
    uint16_t* krow = page_base + (hh * 2 + 0) * (kHalfBytes / 2) + slot * kHeadDim;
    krow[j] = y0;
    krow[j + kHalfDim] = y1;
  };
  if (tid < nk) k_store(tid, k00, k10);
  if (tid + kAppendThreads < nk) k_store(tid + kAppendThreads, k01, k11);
  for (int idx = tid + 2 * kAppendThreads; idx < nk; idx += kAppendThreads) {
    uint16_t k0, k1;
    k_load(idx, k0, k1);
    k_store(idx, k0, k1);
  }
  for (int idx = tid; idx < nv; idx += kAppendThreads) {
    const int hh = idx / (kRowBytes / 16), c = idx - hh * (kRowBytes / 16);
    uint4* vrow = reinterpret_cast<uint4*>(page_base + (hh * 2 + 1) * (kHalfBytes / 2) + slot * kHeadDim);
    vrow[c] = idx == tid ? v0 : vb[idx];
  }
}

constexpr int kPlanThreads = 1024;

// Lists the tiles as {b, first chunk row, tokens, position of the first
// token}: sequence b's chunk gives ceil(len / tokens) tiles. One CTA. The
// tiles are ordered by the number of 64-key steps they take, most first (a
// counting sort over kPlanBuckets buckets, the last one shared by every tile
// of that many steps or more; the order within a bucket is arbitrary), so
// that the CTAs handed out last, as SMs free up, are the short ones. Rows are
// clipped to [0, total); tiles past `capacity` (only possible when chunks
// overlap) are dropped and flagged.
constexpr int kPlanBuckets = 2048;
__device__ void plan_tiles(const int32_t* __restrict__ cu_tokens, const int32_t* __restrict__ start_pos,
                           int batch, int total, int tokens_per_tile, int capacity,
                           int4* __restrict__ tiles, int* __restrict__ num_tiles, int* __restrict__ err) {
  using Scan = cub::BlockScan<int, kPlanThreads>;
  __shared__ typename Scan::TempStorage scan_tmp;
  __shared__ int s_hist[kPlanBuckets];  // tiles per bucket, then the bucket's next slot
  static_assert(kPlanBuckets == 2 * kPlanThreads, "two buckets a thread in the scan");
  for (int k = threadIdx.x; k < kPlanBuckets; k += kPlanThreads) s_hist[k] = 0;
  __syncthreads();
  // a tile's bucket: its steps (from the keys before its last token), most first
  auto bucket = [&](long long pos0, int ntok) {
    if (pos0 < 0 || pos0 > INT_MAX) return kPlanBuckets - 1;  // no work: last
    const long long steps = (pos0 + ntok - 1) / 64 + 1;
    return kPlanBuckets - 1 - static_cast<int>(min(steps, static_cast<long long>(kPlanBuckets - 1)));
  };
  // a warp per sequence, its lanes over the sequence's tiles
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = warp; b < batch; b += kPlanThreads / 32) {
    const int c0 = max(cu_tokens[b], 0), c1 = min(cu_tokens[b + 1], total);
    const int len = c1 - c0;
    if (len <= 0) continue;
    const int nt = (len + tokens_per_tile - 1) / tokens_per_tile;
    for (int j = lane; j < nt; j += 32) {
      const int t0 = j * tokens_per_tile;
      atomicAdd(&s_hist[bucket(static_cast<long long>(start_pos[b]) + t0, min(tokens_per_tile, len - t0))], 1);
    }
  }
  __syncthreads();
  int cnt[2] = {s_hist[2 * threadIdx.x], s_hist[2 * threadIdx.x + 1]}, first[2], all;
  Scan(scan_tmp).ExclusiveSum(cnt, first, all);
  __syncthreads();
  s_hist[2 * threadIdx.x] = first[0];
  s_hist[2 * threadIdx.x + 1] = first[1];
  __syncthreads();
  for (int b = warp; b < batch; b += kPlanThreads / 32) {
    const int c0 = max(cu_tokens[b], 0), c1 = min(cu_tokens[b + 1], total);
    const int len = c1 - c0;
    if (len <= 0) continue;
    const int nt = (len + tokens_per_tile - 1) / tokens_per_tile;
    for (int j = lane; j < nt; j += 32) {
      const int t0 = j * tokens_per_tile, ntok = min(tokens_per_tile, len - t0);
      const long long pos0 = static_cast<long long>(start_pos[b]) + t0;  // -1: does not fit
      const int slot = atomicAdd(&s_hist[bucket(pos0, ntok)], 1);
      if (slot < capacity)
        tiles[slot] = make_int4(b, c0 + t0, ntok, pos0 > INT_MAX ? -1 : static_cast<int>(pos0));
    }
  }
  if (threadIdx.x == 0) {
    if (all > capacity) atomicOr(err, PKV_ERR_SEQ_LEN);
    *num_tiles = min(all, capacity);
  }
}

// The preparation of a prefill call, one launch: block 0 makes the tile plan
// (plan_tiles, the longest part), the other blocks expand the chunk tokens
// (expand_token, one thread a token).
__global__ void __launch_bounds__(kPlanThreads)
    prefill_prep_kernel(int max_blocks, int rope_positions, const int32_t* __restrict__ cu_tokens,
                        const int32_t* __restrict__ start_pos, int batch, int total,
                        int32_t* __restrict__ tok_seq, int32_t* __restrict__ tok_pos,
                        int tokens_per_tile, int capacity, int4* __restrict__ tiles,
                        int* __restrict__ num_tiles, int* __restrict__ err) {
  if (blockIdx.x == 0) {
    plan_tiles(cu_tokens, start_pos, batch, total, tokens_per_tile, capacity, tiles, num_tiles, err);
    return;
  }
  expand_token(static_cast<int>(blockIdx.x - 1) * kPlanThreads + static_cast<int>(threadIdx.x),
               max_blocks, rope_positions, cu_tokens, start_pos, batch, total, tok_seq, tok_pos);
}

struct PrefillAttnParams {
  const float* q_rot;   // [T][hq][64]
  float* out;           // [T][hq][64]
  const int32_t* block_tables;
  int max_blocks;
  long long pos_cap;    // positions at or past this (the block table's or the RoPE table's end) are skipped
  const int4* tiles;
  const int* num_tiles;
  int hkv;
  int hq;
  long long num_pages;
  float qscale;  // scale * log2(e)
  int* err;
};

// ---------------------------------------------------------------------------
// Tensor-core (tcgen05) flash attention for one (tile, kv head).
//
// A tile is TcCfg<G>::kTokens chunk tokens x G query heads = up to 128 rows
// (row R = token R / G, head R % G): the M = 128 of one tcgen05 MMA. Keys go
// in steps of 64 (four pages). Per step j:
//   S_j = Q_hi K_j^T + Q_lo K_j^T    (tensor memory, 128 x 64 fp32, three buffers)
//   softmax warps: P_j = exp2(S_j - m) over S_j's columns, row R = tensor-memory lane R
//   O += P_hi V_j + P_lo V_j         (tensor memory, 128 x 64 fp32; P in tensor memory)
// Q and P enter as bf16 plus their bf16 rounding remainders (each about 16
// bits), as in the decode. The softmax keeps a reference maximum per row and
// moves it (rescaling the row of O in tensor memory) only when a score passes
// it by more than kSlack in the base-2 domain, so P <= 2^kSlack; numerator
// and denominator share the reference, so the result is the same softmax.
// Warps 0-7 (two warpgroups) run the softmax and the epilogue, 16 rows a
// warp and four threads a row (the 16x256b tensor-memory layout; the four
// threads combine row maxima and sums by shuffles); from the second step on
// they make P with the reference as it stands while the row maxima are
// worked out, and make it again in the rare warp whose reference moves.
// Warps 8-11 (one warpgroup, which hands registers to the softmax
// warpgroups) issue: warp 8 the TMA copies of the K rows (each page's 16 K
// rows into the stage's K tile) and warp 11 those of the V rows (into the V
// tile), with separate barriers so K of a later step loads as soon as its
// stage's scores are done, warp 9 the score products and warp 10 the P V
// products. S_j goes out as soon as its buffer and K tile are free, so the
// tensor core computes the next scores while the softmax works on these.
// Every issuing warp runs converged and one elected lane issues (a lone
// thread issuing fell far behind while the softmax warps kept its SM
// sub-partition busy); these warps, normally ahead of the softmax, sleep
// between barrier tests. Every wait is bounded.
template <int G>
struct TcCfg {
  static constexpr int kTokens = 128 / G;
  static constexpr int kRows = kTokens * G;  // <= 128; rows past it are padding
  static constexpr int kStages = 4;
  static constexpr int kSoftmaxThreads = 256;
  static constexpr int kThreads = kSoftmaxThreads + 128;
  // registers a thread after the split (setmaxnreg): the launch gives 80 to
  // each of the 384 threads (two CTAs an SM); the copy and product
  // warpgroup keeps 48, the two softmax warpgroups take 96
  // (128 x 48 + 256 x 96 = 384 x 80)
  static constexpr int kIssueRegs = 48;
  static constexpr int kSoftmaxRegs = 96;
  static_assert(128 * kIssueRegs + kSoftmaxThreads * kSoftmaxRegs <= kThreads * 80,
                "the register shares exceed what two CTAs an SM give a CTA");
  static constexpr uint32_t kTile = 128 * 128;  // a 128-row x 128-byte operand tile
  static constexpr uint32_t kStep = 64 * 128;   // 64 K rows (or V rows) of one step
  // dynamic shared memory: Q_hi, Q_lo, then per stage K and V
  static constexpr uint32_t kQhi = 0, kQlo = kTile;
  static constexpr uint32_t kStage0 = 2 * kTile;
  static constexpr uint32_t kBytes = kStage0 + kStages * 2 * kStep;
};
constexpr float kSlack = 8.f;
// tensor memory: three S buffers in columns 0-63, 64-127 and 128-191 (step j
// uses buffer j % 3), O in 192-255. Step j's P is written over its own S:
// P_hi in the buffer's first 32 columns and P_lo in the next 32 (two bf16
// keys per column). A softmax step does not wait for the previous step's
// P V (only to rescale O), and S_j goes into the buffer of P_{j-3}, whose
// product is normally long done.
constexpr int kSBufs = 3;
constexpr uint32_t kTmemCols = 256;

// Two fp32 values in one 64-bit register, and the paired fp32 arithmetic of
// sm_100 and later (each half rounded exactly as the scalar operation).
__device__ __forceinline__ uint64_t f32x2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return make_float2(a, b);
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Bounded wait for the copy and product warps, which are normally ahead of
// the softmax: after a first test, they sleep between tests instead of
// polling, so that their spinning does not take issue slots from the softmax
// warps on the same sub-partition.
__device__ __forceinline__ bool mbar_wait_idle(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    __nanosleep(32);
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}

// p0 - h.lo and p1 - h.hi for the two bf16 halves of h, each in one
// mixed-precision fma (bf16 times bf16 -1, plus fp32; sm_100 and later):
// exact when h is p rounded to bf16, so the remainder of the split
__device__ __forceinline__ float2 bf16x2_remainder(uint32_t h, float p0, float p1) {
  float r0, r1;
  asm("{\n\t.reg .b16 h0, h1, m1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "mov.b16 m1, 0xBF80;\n\t"
      "fma.rn.f32.bf16 %0, h0, m1, %3;\n\t"
      "fma.rn.f32.bf16 %1, h1, m1, %4;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "r"(h), "f"(p0), "f"(p1));
  return make_float2(r0, r1);
}

// Move registers between the warpgroups of a CTA (every warp of a warpgroup
// executes the same instruction): dec gives back down to N a thread, inc
// waits until N a thread are free.
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// max of three floats in one instruction (sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int G>
__global__ void __launch_bounds__(TcCfg<G>::kThreads, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kv16_map, const PrefillAttnParams p) {
  using C = TcCfg<G>;
  extern __shared__ __align__(1024) uint8_t dsmem[];
  __shared__ __align__(8) uint64_t k_full[C::kStages], k_empty[C::kStages];
  __shared__ __align__(8) uint64_t v_full[C::kStages], v_empty[C::kStages];
  __shared__ __align__(8) uint64_t s_full[kSBufs], q_ready, p_full[kSBufs], pv_done[kSBufs], drain[2];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA x works on tile x / hkv for kv head x % hkv: the hardware hands CTAs
  // out in order of x, so the order of the tiles (most steps first) holds
  // across all kv heads
  const int ti = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.hkv));
  const int h = static_cast<int>(blockIdx.x - static_cast<unsigned>(ti) * static_cast<unsigned>(p.hkv));
  if (ti >= *p.num_tiles) return;
  const int4 tile = p.tiles[ti];
  const int b = tile.x, row0 = tile.y, n_tok = tile.z, pos0 = tile.w;
  const long long room = p.pos_cap - pos0;
  const int n_ok = pos0 < 0 ? 0 : static_cast<int>(min(static_cast<long long>(n_tok), max(room, 0ll)));
  for (int e = n_ok * G * kHeadDim + tid; e < n_tok * G * kHeadDim; e += C::kThreads) {
    const int t = e / (G * kHeadDim), rest = e - t * (G * kHeadDim);
    p.out[(static_cast<size_t>(row0 + t) * p.hq + h * G) * kHeadDim + rest] = 0.f;
  }
  if (n_ok <= 0) return;
  const int last_pos = pos0 + n_ok - 1;
  const int n_pages = last_pos / kPage + 1;
  const int n_steps = (n_pages + 3) / 4;
  const int32_t* bt = p.block_tables + static_cast<size_t>(b) * p.max_blocks;
  const uint32_t base = (smem_addr(dsmem) + 1023u) & ~1023u;
  uint8_t* gbase = dsmem + (base - smem_addr(dsmem));
  auto kst = [&](int st) { return base + C::kStage0 + st * 2 * C::kStep; };
  auto vst = [&](int st) { return base + C::kStage0 + st * 2 * C::kStep + C::kStep; };

  if (warp == 0) {
    tmem_alloc(smem_addr(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(smem_addr(&k_full[st]), 1);
      mbar_init(smem_addr(&k_empty[st]), 1);
      mbar_init(smem_addr(&v_full[st]), 1);
      mbar_init(smem_addr(&v_empty[st]), 1);
    }
    mbar_init(smem_addr(&q_ready), C::kSoftmaxThreads);
    // S_j done, P_j ready and P_j V_j done, one barrier each per buffer
    // (j % 3): a wait for step j never sees its barrier two phases on
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(smem_addr(&s_full[i]), 1);
      mbar_init(smem_addr(&p_full[i]), C::kSoftmaxThreads);
      mbar_init(smem_addr(&pv_done[i]), 1);
    }
    mbar_init(smem_addr(&drain[0]), 1);
    mbar_init(smem_addr(&drain[1]), 1);
  }
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Everything above (the tile, the zeroed rows, tensor memory and the
  // barriers) overlaps the end of the append kernel before this one; the
  // rotated queries and the pool pages it writes are read only from here on.
  grid_dependency_wait();
  const uint32_t tmem = s_tmem, tO = tmem + 64 * kSBufs;
  auto tS = [&](int j) { return tmem + 64 * (j % kSBufs); };  // S_j, then P_j (hi: +0, lo: +32)
  auto buf = [](int j) { return j % kSBufs; };                   // step j's S / P / P V barriers
  auto par = [](int j) { return static_cast<uint32_t>((j / kSBufs) & 1); };  // and their phase parity
  bool failed = false;

  if (warp >= 8) {
    // the copy and product warps (one warpgroup) give registers to the
    // softmax warpgroups, first thing and unconditionally, so the softmax
    // warps' increase (the shares add up to the launch's total) never waits
    // for more than this
    regs_dec<TcCfg<G>::kIssueRegs>();
    if (warp == 8 || warp == 11) {
      // ---- TMA producers, warp 8 for K and warp 11 for V: step j's four
      // pages into stage j % kStages. A warp reads the page ids 32 at a time
      // (lane i: page 32 m + i), the next 32 while it issues the current ones,
      // so no step waits for a block-table load; the whole warp runs the loop
      // and one elected lane issues each copy. K and V have a warp each so
      // that the K copies, needed first, never queue behind a wait for a V
      // stage. ----
      const int kind = warp == 8 ? 0 : 1;  // 0: K rows, 1: V rows
      uint64_t* full = kind ? v_full : k_full;
      uint64_t* empty = kind ? v_empty : k_empty;
      int issued = 0;
      // lane i: the copy's row coordinate for page 32 m + i of window m (-1:
      // past the last page, or a bad id), and the window's valid pages as a
      // bit mask; worked out once per window of eight steps
      uint32_t valid = 0;
      auto window = [&](int pid, int m) {
        const int pg = 32 * m + lane;
        const bool in = pg < n_pages;
        const bool ok = in && pid >= 0 && static_cast<long long>(pid) < p.num_pages;
        if (kind == 0 && __any_sync(kFull, in && !ok) && lane == 0) atomicOr(p.err, PKV_ERR_PAGE_ID);
        valid = __ballot_sync(kFull, ok);
        return ok ? (pid * p.hkv + h) * (2 * kPage) + kind * kPage : -1;
      };
      int row = window(lane < n_pages ? bt[lane] : -1, 0);
      int pid_next = 32 + lane < n_pages ? bt[32 + lane] : -1;
      for (int j = 0; j < n_steps && !failed; ++j) {
        const int st = j % C::kStages, use = j / C::kStages;
        if (j > 0 && (j & 7) == 0) {  // the next 32 pages
          row = window(pid_next, j >> 3);
          const int nxt = 4 * j + 32 + lane;
          pid_next = nxt < n_pages ? bt[nxt] : -1;
        }
        const int l0 = (4 * j) & 31;
        const uint32_t vbits = (valid >> l0) & 0xFu;
        int rows[4];
  #pragma unroll
        for (int q = 0; q < 4; ++q) rows[q] = __shfl_sync(kFull, row, l0 + q);
        // the stage is free once its scores (K) or its P V product (V) are done
        if (use > 0 && !mbar_wait_idle(smem_addr(&empty[st]), (use - 1) & 1)) failed = true;
        if (__any_sync(kFull, failed)) {
          failed = true;
          break;
        }
        const uint32_t dst = (kind ? vst(st) : kst(st)), bar = smem_addr(&full[st]);
        mbar_arrive_expect_tx_elect(bar, static_cast<uint32_t>(__popc(vbits)) * kHalfBytes);
  #pragma unroll
        for (int q = 0; q < 4; ++q)
          if ((vbits >> q) & 1u) tma_load_2d_elect(dst + q * kHalfBytes, &kv16_map, 0, rows[q], bar);
        issued = j + 1;
      }
      // let the copies still in flight (the last kStages steps at most) land
      // before shared memory goes away
      if (failed && lane == 0)
        for (int j = max(0, issued - C::kStages); j < issued; ++j)
          mbar_wait_bounded(smem_addr(&full[j % C::kStages]), (j / C::kStages) & 1);
    } else {
      // ---- MMA issuers, each a whole warp, converged (one lane issues each
      // product; every wait's result is made warp-uniform): warp 9 the score
      // products, warp 10 the P V products. A commit covers only its own
      // warp's products. ----
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(kFull, mbar_wait_idle(bar, parity)) != 0;
      };
      if (warp == 9) {
        constexpr uint32_t idS = idesc_bf16_f32(128, 64, false);
        const uint64_t dQhi = smem_desc_sw128(base + C::kQhi), dQlo = smem_desc_sw128(base + C::kQlo);
        if (!wait_all(smem_addr(&q_ready), 0)) failed = true;
        for (int j = 0; j < n_steps && !failed; ++j) {
          const int st = j % C::kStages;
          // S_j goes into the buffer of P_{j-3}: once P_{j-3} V_{j-3} is done
          if (j >= kSBufs && !wait_all(smem_addr(&pv_done[buf(j)]), par(j - kSBufs))) failed = true;
          if (failed || !wait_all(smem_addr(&k_full[st]), (j / C::kStages) & 1)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t dK = smem_desc_sw128(kst(st));
          // K-major tiles: a 16-element K step is 32 bytes along the swizzled
          // row (+2 in the descriptor's 16-byte address units)
  #pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16(tS(j), dQhi + 2 * k, dK + 2 * k, idS, k > 0);
  #pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16(tS(j), dQlo + 2 * k, dK + 2 * k, idS, true);
          umma_commit(smem_addr(&k_empty[st]));
          umma_commit(smem_addr(&s_full[buf(j)]));
        }
      } else {
        constexpr uint32_t idPV = idesc_bf16_f32(128, 64, true);
        for (int j = 0; j < n_steps && !failed; ++j) {
          const int st = j % C::kStages;
          if (!wait_all(smem_addr(&p_full[buf(j)]), par(j)) ||
              !wait_all(smem_addr(&v_full[st]), (j / C::kStages) & 1)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint64_t dV = smem_desc_sw128(vst(st));
          // P from tensor memory (a 16-key K step is 8 columns); V is MN-major:
          // a 16-key K step is 16 rows = 2048 bytes (+128)
  #pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16_tmem_a(tO, tS(j) + 8 * k, dV + 128 * k, idPV, j > 0 || k > 0);
  #pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16_tmem_a(tO, tS(j) + 32 + 8 * k, dV + 128 * k, idPV, true);
          umma_commit(smem_addr(&v_empty[st]));
          umma_commit(smem_addr(&pv_done[buf(j)]));
        }
      }
      if (failed) {  // let this warp's products already issued finish before the memory goes away
        umma_commit(smem_addr(&drain[warp - 9]));
        mbar_wait_bounded(smem_addr(&drain[warp - 9]), 0);
      }
    }
  } else {
    regs_inc<TcCfg<G>::kSoftmaxRegs>();
    // ---- softmax and epilogue. Warp w owns rows L .. L + 15, L = 32 (w % 4)
    // + 16 (w / 4) (tensor-memory lanes). Its thread t holds rows L + t / 4
    // (hh = 0) and L + t / 4 + 8 (hh = 1) and, of each, the key pairs
    // 8 i + 2 q and 8 i + 2 q + 1 (i = 0..7, q = t % 4): the 16x256b layout,
    // in which S word 4 i + 2 hh + e is key 8 i + 2 q + e of row hh. The four
    // threads of a row are lanes of one warp, so row maxima and sums combine
    // by shuffles, and the warp's reads of S_j are done before its P_j stores
    // over the same columns.
    const int q = lane & 3;
    const int lrow = 32 * (warp & 3) + 16 * (warp >> 2);  // the warp's first row
    const uint32_t lane_addr = static_cast<uint32_t>(lrow) << 16;
    int tok[2], gix[2], pos[2];
    bool live[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int rw = lrow + (lane >> 2) + 8 * hh;
      tok[hh] = rw / G;
      gix[hh] = rw - tok[hh] * G;
      live[hh] = rw < C::kRows && tok[hh] < n_ok;
      pos[hh] = pos0 + min(tok[hh], n_ok - 1);
    }
    // Q rows: scaled, as bf16 high part and remainder, 128-byte swizzled
    // (this thread: dims 16 q .. 16 q + 15 of its two rows, chunks 2 q and 2 q + 1)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int rw = lrow + (lane >> 2) + 8 * hh;
      const float* qr =
          p.q_rot + (static_cast<size_t>(row0 + (live[hh] ? tok[hh] : 0)) * p.hq + h * G + gix[hh]) * kHeadDim + 16 * q;
      float x[16];
#pragma unroll
      for (int d = 0; d < 16; d += 4) {
        const float4 v = live[hh] ? *reinterpret_cast<const float4*>(qr + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        x[d] = v.x * p.qscale;
        x[d + 1] = v.y * p.qscale;
        x[d + 2] = v.z * p.qscale;
        x[d + 3] = v.w * p.qscale;
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * q + cc;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = x[8 * cc + 2 * e], a1 = x[8 * cc + 2 * e + 1];
          hi[e] = pack_bf16x2(a0, a1);
          const float2 f = bf16x2_to_float2(hi[e]);
          lo[e] = pack_bf16x2(a0 - f.x, a1 - f.y);
        }
        const uint32_t off = rw * 128 + ((c ^ (rw & 7)) << 4);
        *reinterpret_cast<uint4*>(gbase + C::kQhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(gbase + C::kQlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(smem_addr(&q_ready));

    float m_ref[2] = {-INFINITY, -INFINITY}, l_sum[2] = {0.f, 0.f};
    // which pages have a bad id: bit i of bad_win for page 32 m + i, from the
    // warp's window of page ids (lane i reads page 32 m + i), the next window
    // loaded while this one is used
    auto bad_bits = [&](int m) {
      const int pg = 32 * m + lane;
      const int page = pg < n_pages ? bt[pg] : 0;
      return __ballot_sync(kFull, pg < n_pages && (page < 0 || static_cast<long long>(page) >= p.num_pages));
    };
    uint32_t bad_win = bad_bits(0), bad_nextwin = n_pages > 32 ? bad_bits(1) : 0u;
    for (int j = 0; j < n_steps; ++j) {
      const int st = j % C::kStages;
      const int kb = 64 * j + 2 * q;  // key position of this thread's first key
      if (j > 0 && (j & 7) == 0) {
        bad_win = bad_nextwin;
        bad_nextwin = 32 * (j / 8 + 1) < n_pages ? bad_bits(j / 8 + 1) : 0u;
      }
      const int bad = static_cast<int>((bad_win >> ((4 * j) & 31)) & 0xFu);
      if (!mbar_wait_bounded(smem_addr(&s_full[buf(j)]), par(j))) failed = true;
      tc_fence_after();
      // S_j, with the keys that get no weight (past the row's position, or
      // of a page with a bad id: page i / 2 of the step holds pair i) at -inf
      float sv[32];
      auto load_s = [&]() {
        tmem_ld_16x256b_x8(tS(j) + lane_addr, sv);
        tmem_wait_ld();
        if (64 * j + 63 > pos[0] || bad) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
              for (int e = 0; e < 2; ++e)
                if (kb + 8 * i + e > pos[hh] || ((bad >> (i >> 1)) & 1)) sv[4 * i + 2 * hh + e] = -INFINITY;
        }
      };
      // P = exp2(S - m_ref) as bf16 high part and remainder, into tensor
      // memory over S_j (16x128b: word 2 i + hh is column 4 i + q, the pair
      // 8 i + 2 q, + 1 of row hh; P_hi in columns 0-31, P_lo in 32-63), in
      // paired fp32 arithmetic, with the row sums and, alongside, this
      // thread's maximum of each of its rows (three-input maxima)
      uint32_t hi[16], lo[16];
      uint64_t lp[2];
      float mt[2];
      auto make_p = [&]() {
        uint64_t mm[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float m_use = m_ref[hh] == -INFINITY ? 0.f : m_ref[hh];  // all scores -inf: P = 0
          mm[hh] = f32x2(m_use, m_use);
          lp[hh] = f32x2(0.f, 0.f);
          mt[hh] = -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int w = 4 * i + 2 * hh;
            mt[hh] = fmax3(mt[hh], sv[w], sv[w + 1]);
            const float2 d = unpack_f32x2(sub_f32x2(f32x2(sv[w], sv[w + 1]), mm[hh]));
            const float p0 = fast_exp2(d.x), p1 = fast_exp2(d.y);
            lp[hh] = add_f32x2(lp[hh], f32x2(p0, p1));
            hi[2 * i + hh] = pack_bf16x2(p0, p1);
            const float2 rem = bf16x2_remainder(hi[2 * i + hh], p0, p1);
            lo[2 * i + hh] = pack_bf16x2(rem.x, rem.y);
          }
      };
      // From the second step on, where the reference rarely moves, P is made
      // with the reference as it stands, before the row maxima are known, so
      // that the maxima's shuffles overlap the exponentials; a warp where a
      // row's reference moves drops it and makes P again from S_j, still in
      // tensor memory. The first step takes the maxima first.
      const bool spec = j > 0;
      load_s();
      if (spec) {
        make_p();
      } else {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          mt[hh] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 8; ++i) mt[hh] = fmax3(mt[hh], sv[4 * i + 2 * hh], sv[4 * i + 2 * hh + 1]);
        }
      }
      // each row's maximum: the row's four threads (lanes 4 (t / 4) .. + 3)
      float mx[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float m = fmaxf(mt[hh], __shfl_xor_sync(kFull, mt[hh], 1));
        mx[hh] = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
      }
      // Move the reference up where a score passed it by more than kSlack;
      // O and l follow, O once P_{j-1} V_{j-1}, the last product into it, is
      // done. The tensor-memory loads and stores are warp-wide, so a warp
      // rescales O when any of its rows moves, the other rows by exactly 1.
      bool moves[2], resc[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        moves[hh] = mx[hh] > m_ref[hh] + kSlack;
        resc[hh] = moves[hh] && j > 0 && m_ref[hh] != -INFINITY;
      }
      if (__any_sync(kFull, moves[0] || moves[1])) {  // a speculative P is dropped
        if (__any_sync(kFull, resc[0] || resc[1])) {
          if (!mbar_wait_bounded(smem_addr(&pv_done[buf(j - 1)]), par(j - 1))) failed = true;
          tc_fence_after();
          uint64_t aa[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float alpha = resc[hh] ? fast_exp2(m_ref[hh] - mx[hh]) : 1.f;
            l_sum[hh] *= alpha;
            aa[hh] = f32x2(alpha, alpha);
          }
          float o[32];
          tmem_ld_16x256b_x8(tO + lane_addr, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int w = 4 * i + 2 * hh;
              const float2 v = unpack_f32x2(mul_f32x2(f32x2(o[w], o[w + 1]), aa[hh]));
              o[w] = v.x;
              o[w + 1] = v.y;
            }
          tmem_st_16x256b_x8(tO + lane_addr, o);
          tmem_wait_st();
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          if (moves[hh]) m_ref[hh] = mx[hh];
        if (spec) load_s();
        make_p();
      } else if (!spec) {
        make_p();
      }
      tmem_st_16x128b_x8(tS(j) + lane_addr, hi);
      tmem_st_16x128b_x8(tS(j) + lane_addr + 32, lo);
      tmem_wait_st();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float2 a = unpack_f32x2(lp[hh]);
        l_sum[hh] += a.x + a.y;
      }
      // V rows that hold no key of the tile (past its last position, or of a
      // page with a bad id) are zeroed once the stage's V copies have landed,
      // so that their bits cannot reach O
      if (64 * j + 63 > last_pos || bad) {
        if (!mbar_wait_bounded(smem_addr(&v_full[st]), (j / C::kStages) & 1)) failed = true;
        uint8_t* vrow = gbase + (vst(st) - base);
        for (int idx = tid; idx < 64 * 8; idx += C::kSoftmaxThreads) {
          const int key = idx >> 3;
          if (64 * j + key > last_pos || ((bad >> (key >> 4)) & 1))
            *reinterpret_cast<uint4*>(vrow + key * 128 + (idx & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the zeroed rows, before the tensor core reads V
      }
      tc_fence_before();
      mbar_arrive(smem_addr(&p_full[buf(j)]));
    }
    // epilogue: O / l for the live rows, l summed over the row's four threads.
    // The last product into O is P V of step n_steps - 1 (the one before it
    // on the same barrier, of step n_steps - 1 - kSBufs, was done before S of
    // step n_steps - 1 was issued). The decision is warp-uniform: the
    // tensor-memory load below is warp-wide.
    const bool done = !failed && mbar_wait_bounded(smem_addr(&pv_done[buf(n_steps - 1)]), par(n_steps - 1));
    if (__all_sync(kFull, done)) {
      tc_fence_after();
      float o[32];
      tmem_ld_16x256b_x8(tO + lane_addr, o);
      tmem_wait_ld();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float l = l_sum[hh];
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        if (live[hh]) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          float* dst = p.out + (static_cast<size_t>(row0 + tok[hh]) * p.hq + h * G + gix[hh]) * kHeadDim + 2 * q;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float2*>(dst + 8 * i) =
                make_float2(o[4 * i + 2 * hh] * inv, o[4 * i + 2 * hh + 1] * inv);
        }
      }
    } else {
      failed = true;
    }
  }
  if (failed && lane == 0) atomicOr(p.err, PKV_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Workspace: each chunk token's sequence and position, then the tile list
// and its count.
struct PrefillLayout {
  size_t seq, pos, tiles, count, total;
};

// An upper bound on the tiles of any split of total_tokens over the batch
// (at most one partial tile per sequence); tokens per tile are at least 16.
size_t max_tiles(int total_tokens, int batch) {
  return static_cast<size_t>(total_tokens) / 16 + static_cast<size_t>(batch) + 1;
}

PrefillLayout layout(int total_tokens, int batch, int max_blocks) {
  (void)max_blocks;
  PrefillLayout l;
  l.seq = 0;
  l.pos = l.seq + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens));
  l.tiles = l.pos + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens));
  l.count = l.tiles + align256(sizeof(int4) * max_tiles(total_tokens, batch));
  l.total = l.count + 256;
  return l;
}

// The three launches of a prefill call for groups of G query heads: the
// preparation (token expansion and tile plan), the append, the attention.
template <int G>
cudaError_t launch_all(const PrefillLaunch& a, const PrefillLayout& l, cudaStream_t stream) {
  using C = TcCfg<G>;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int32_t* tok_seq = reinterpret_cast<int32_t*>(ws + l.seq);
  int32_t* tok_pos = reinterpret_cast<int32_t*>(ws + l.pos);
  int4* tiles = reinterpret_cast<int4*>(ws + l.tiles);
  int* count = reinterpret_cast<int*>(ws + l.count);
  const size_t grid_x = static_cast<size_t>(a.total_tokens + C::kTokens - 1) / C::kTokens + a.batch;
  const int expand_blocks = (a.total_tokens + kPlanThreads - 1) / kPlanThreads;
  prefill_prep_kernel<<<1 + expand_blocks, kPlanThreads, 0, stream>>>(
      a.max_blocks, a.rope_positions, a.cu_tokens, a.start_pos, a.batch, a.total_tokens, tok_seq,
      tok_pos, C::kTokens, static_cast<int>(grid_x), tiles, count, a.err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the caller's RoPE table: fp32 pair rows, then fp64 rows, one per position
  const float4* rope_ff = static_cast<const float4*>(a.rope_table);
  const double2* rope_dd =
      reinterpret_cast<const double2*>(rope_ff + static_cast<size_t>(a.rope_positions) * kHalfDim);
  prefill_append_kernel<<<a.total_tokens, kAppendThreads, 0, stream>>>(
      const_cast<uint16_t*>(reinterpret_cast<const uint16_t*>(a.pool)), a.num_pages, a.num_kv_heads,
      a.num_q_heads, a.q, a.k, a.v, a.q_rot, a.block_tables, a.max_blocks, tok_seq, tok_pos, rope_ff,
      rope_dd, a.err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  PrefillAttnParams p;
  p.q_rot = a.q_rot;
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.max_blocks = a.max_blocks;
  p.pos_cap = static_cast<long long>(a.max_blocks) * kPage < a.rope_positions
                  ? static_cast<long long>(a.max_blocks) * kPage
                  : static_cast<long long>(a.rope_positions);
  p.tiles = tiles;
  p.num_tiles = count;
  p.hkv = a.num_kv_heads;
  p.hq = a.num_q_heads;
  p.num_pages = a.num_pages;
  p.qscale = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.err = a.err;
  const int smem = static_cast<int>(C::kBytes + 1024);  // + alignment to 1 KiB
  static std::atomic<bool> attr_set[9];
  if (!attr_set[G].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // The warpgroups' register shares must fit in what the launch gives the
    // CTA (the compiler's count a thread x its threads), or the softmax
    // warps' increase would wait for registers that never come: refuse.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, prefill_tc_kernel<G>);
    if (e != cudaSuccess) return e;
    if (128 * C::kIssueRegs + C::kSoftmaxThreads * C::kSoftmaxRegs > C::kThreads * fa.numRegs)
      return cudaErrorInvalidConfiguration;
    attr_set[G].store(true, std::memory_order_relaxed);
  }
  const size_t n_ctas = grid_x * static_cast<size_t>(a.num_kv_heads);
  if (n_ctas > 0x7fffffffu) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(n_ctas));
  // programmatic dependent launch: the kernel's set-up overlaps the append's end
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<G>, *a.kv16_map, p);
}

}  // namespace

size_t prefill_workspace_bytes(int total_tokens, int batch, int max_blocks) {
  return layout(total_tokens, batch, max_blocks).total;
}

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t stream) {
  if (a.total_tokens == 0) return cudaSuccess;
  const PrefillLayout l = layout(a.total_tokens, a.batch, a.max_blocks);

  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_all<1>(a, l, stream);
    case 2: return launch_all<2>(a, l, stream);
    case 3: return launch_all<3>(a, l, stream);
    case 4: return launch_all<4>(a, l, stream);
    case 5: return launch_all<5>(a, l, stream);
    case 6: return launch_all<6>(a, l, stream);
    case 7: return launch_all<7>(a, l, stream);
    case 8: return launch_all<8>(a, l, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
