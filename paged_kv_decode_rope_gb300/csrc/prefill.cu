// prefill.cu -- chunked causal prefill into the page pool.
//
// "Hours of YouTube and 85 handtyped pages of notes on LLM Inference – Start
// here": prefill fills the prompt pages (dense causal prefill), decode then
// appends one token at a time. A chunk of new tokens for sequence b sits at
// positions start_pos[b], start_pos[b]+1, ...; every chunk token is rotated
// and appended like a decode token, and the queries of chunk token t attend
// causally over the sequence's first start_pos[b] + t + 1 tokens.
//
// Three launches. (1) An expansion kernel turns every chunk token into a
// one-token "virtual sequence" (its causal length, its position, its
// sequence's block table row). (2) The append kernel rotates and stores every
// chunk token exactly as it does a decode token, and writes the rotated
// queries. (3) A flash-attention kernel on tensor cores: one CTA per
// (sequence, kv head, tile of query tokens) streams the sequence's pages up
// to the tile's last position through a shared-memory ring (one TMA copy per
// page) and every warp runs 16 (token, query head) rows of the tile against
// each page: S = Q K^T and O += P V as m16n8k16 bf16 products with fp32
// accumulation, the causal mask on the pages that hold the tile's positions,
// and an online softmax per row. Q and P go in as bf16 plus a second product
// with their bf16 rounding remainders, so both carry about 16 bits, as in the
// decode. A tile plan (one CTA) lists the (sequence, first token) of every
// tile.
#include <cerrno>
#include <climits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kExpandThreads = 128;

// One CTA per chunk token: find its sequence by bisection over cu_tokens,
// then write its length (0 when the sequence's chunk is malformed: the
// append and decode then flag it and zero its rows), its position, and a
// copy of its sequence's block table row.
__global__ void prefill_expand_kernel(const int32_t* __restrict__ block_tables, int max_blocks,
                                      const int32_t* __restrict__ cu_tokens,
                                      const int32_t* __restrict__ start_pos, int batch, int total,
                                      int32_t* __restrict__ tok_tables, int32_t* __restrict__ tok_lens,
                                      int32_t* __restrict__ tok_pos) {
  const int idx = blockIdx.x;
  if (idx >= total) return;
  int lo = 0, hi = batch - 1;  // largest b with cu_tokens[b] <= idx
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_tokens[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int c0 = cu_tokens[b], c1 = cu_tokens[b + 1];
  const long long pos = static_cast<long long>(start_pos[b]) + (idx - c0);
  const bool ok = c0 <= idx && idx < c1 && start_pos[b] >= 0 &&
                  pos + 1 <= static_cast<long long>(max_blocks) * kPage;
  if (threadIdx.x == 0) {
    tok_lens[idx] = ok ? static_cast<int32_t>(pos + 1) : 0;
    tok_pos[idx] = ok ? static_cast<int32_t>(pos) : 0;
  }
  const int32_t* src = block_tables + static_cast<size_t>(b) * max_blocks;
  int32_t* dst = tok_tables + static_cast<size_t>(idx) * max_blocks;
  for (int i = threadIdx.x; i < max_blocks; i += kExpandThreads) dst[i] = src[i];
}

// Query tokens per tile: 32 for groups of up to 4 query heads, 16 above,
// so a CTA has 2G or G warps of 16 (token, head) rows each.
template <int G>
struct PrefillCfg {
  static constexpr int kTokens = G <= 4 ? 32 : 16;
  static constexpr int kRows = kTokens * G;
  static constexpr int kWarps = kRows / 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStages = 4;
};
constexpr int kPlanThreads = 1024;

// Lists the tiles as {b, first chunk row, tokens, position of the first
// token}: sequence b's chunk gives ceil(len / tokens) tiles. One CTA; slots
// are reserved with a shared-memory counter, so sequences land in arbitrary
// order (tiles are independent); within a sequence the last tile, which reads
// the most pages, goes first. Rows are clipped to [0, total); tiles past
// `capacity` (only possible when chunks overlap) are dropped and flagged.
__global__ void prefill_plan_kernel(const int32_t* __restrict__ cu_tokens,
                                    const int32_t* __restrict__ start_pos, int batch, int total,
                                    int tokens_per_tile, int capacity, int4* __restrict__ tiles,
                                    int* __restrict__ num_tiles, int* __restrict__ err) {
  __shared__ int s_count;
  if (threadIdx.x == 0) s_count = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < batch; b += kPlanThreads) {
    const int c0 = max(cu_tokens[b], 0), c1 = min(cu_tokens[b + 1], total);
    const int len = c1 - c0;
    if (len <= 0) continue;
    const int nt = (len + tokens_per_tile - 1) / tokens_per_tile;
    const int base = atomicAdd(&s_count, nt);
    for (int i = 0; i < nt; ++i) {
      const int j = nt - 1 - i, t0 = j * tokens_per_tile;
      const long long pos0 = static_cast<long long>(start_pos[b]) + t0;  // -1: does not fit
      if (base + i < capacity)
        tiles[base + i] = make_int4(b, c0 + t0, min(tokens_per_tile, len - t0),
                                    pos0 > INT_MAX ? -1 : static_cast<int>(pos0));
    }
    if (base + nt > capacity) atomicOr(err, PKV_ERR_SEQ_LEN);
  }
  __syncthreads();
  if (threadIdx.x == 0) *num_tiles = min(s_count, capacity);
}

struct PrefillAttnParams {
  const float* q_rot;   // [T][hq][64]
  float* out;           // [T][hq][64]
  const int32_t* block_tables;
  int max_blocks;
  const int4* tiles;
  const int* num_tiles;
  int hkv;
  int hq;
  long long num_pages;
  float qscale;  // scale * log2(e)
  int* err;
};

// Flash attention for one (tile, kv head): blockIdx.x = tile, blockIdx.y = kv head.
template <int G>
__global__ void __launch_bounds__(PrefillCfg<G>::kThreads)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap kv_map, const PrefillAttnParams p) {
  using C = PrefillCfg<G>;
  __shared__ __align__(1024) uint8_t ring[C::kStages][kHeadPageBytes];
  __shared__ __align__(8) uint64_t full_bar[C::kStages], empty_bar[C::kStages];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, tig = lane & 3, mi = lane >> 3, ri = lane & 7;
  if (static_cast<int>(blockIdx.x) >= *p.num_tiles) return;  // the grid is an upper bound
  const int4 tile = p.tiles[blockIdx.x];
  const int b = tile.x, row0 = tile.y, n_tok = tile.z, pos0 = tile.w, h = blockIdx.y;
  // Tokens whose position does not fit the block table (the append flagged
  // them) get zero rows; the rest of the tile is attended as usual.
  const long long room = static_cast<long long>(p.max_blocks) * kPage - pos0;
  const int n_ok = pos0 < 0 ? 0 : static_cast<int>(min(static_cast<long long>(n_tok), max(room, 0ll)));
  for (int e = n_ok * G * kHeadDim + tid; e < n_tok * G * kHeadDim; e += C::kThreads) {
    const int t = e / (G * kHeadDim), rest = e - t * (G * kHeadDim);
    p.out[(static_cast<size_t>(row0 + t) * p.hq + h * G) * kHeadDim + rest] = 0.f;
  }
  if (n_ok <= 0) return;
  const int last_pos = pos0 + n_ok - 1;
  const int n_pages = last_pos / kPage + 1;
  const int32_t* bt = p.block_tables + static_cast<size_t>(b) * p.max_blocks;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), C::kWarps);
    }
  }
  fence_mbar_init();
  __syncthreads();

  // thread 0 fills stage s with page pg (one 4 KiB box: 16 K rows, then 16 V rows)
  int issued = 0;  // pages thread 0 has started copying
  auto issue = [&](int pg, int s) {
    ++issued;
    const int page = bt[pg];
    const uint32_t bar = smem_addr(&full_bar[s]);
    if (page < 0 || static_cast<long long>(page) >= p.num_pages) {
      atomicOr(p.err, PKV_ERR_PAGE_ID);
      mbar_arrive(bar);  // nothing to wait for; the stage keeps stale rows
      return;
    }
    mbar_arrive_expect_tx(bar, kHeadPageBytes);
    // default L2 policy: the other tiles of the sequence read the same pages
    tma_load_2d(smem_addr(ring[s]), &kv_map, 0, (page * p.hkv + h) * (2 * kPage), bar);
  };
  if (tid == 0)
    for (int s = 0; s < C::kStages && s < n_pages; ++s) issue(s, s);

  // This lane's two rows: R = 16 warp + g8 (+8) -> token R / G, query head h G + R % G.
  int pos[2];
  bool live[2];
  uint32_t qh[4][4], ql[4][4];  // Q hi / lo as the A operand, per 16-dim k-step
  {
    float x[2][4][4];  // [row][k-step][c]: dims 16s + 2tig + {0,1}, 16s + 8 + 2tig + {0,1}
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int R = 16 * warp + g8 + 8 * rr;
      const int t = R / G, i = R - t * G;
      live[rr] = t < n_ok;
      pos[rr] = pos0 + min(t, n_ok - 1);  // rows past the tile copy its last position
      const float* qr =
          p.q_rot + (static_cast<size_t>(row0 + (live[rr] ? t : 0)) * p.hq + h * G + i) * kHeadDim;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const float2 a = *reinterpret_cast<const float2*>(qr + 16 * s + 2 * tig);
        const float2 c = *reinterpret_cast<const float2*>(qr + 16 * s + 8 + 2 * tig);
        x[rr][s][0] = a.x * p.qscale;
        x[rr][s][1] = a.y * p.qscale;
        x[rr][s][2] = c.x * p.qscale;
        x[rr][s][3] = c.y * p.qscale;
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      // a0: row g8, dims 2tig..; a1: row g8+8; a2: row g8, dims 8+2tig..; a3: row g8+8
      const uint32_t h0 = pack_bf16x2(x[0][s][0], x[0][s][1]), h1 = pack_bf16x2(x[1][s][0], x[1][s][1]);
      const uint32_t h2 = pack_bf16x2(x[0][s][2], x[0][s][3]), h3 = pack_bf16x2(x[1][s][2], x[1][s][3]);
      qh[s][0] = h0; qh[s][1] = h1; qh[s][2] = h2; qh[s][3] = h3;
      const float2 f0 = bf16x2_to_float2(h0), f1 = bf16x2_to_float2(h1);
      const float2 f2 = bf16x2_to_float2(h2), f3 = bf16x2_to_float2(h3);
      ql[s][0] = pack_bf16x2(x[0][s][0] - f0.x, x[0][s][1] - f0.y);
      ql[s][1] = pack_bf16x2(x[1][s][0] - f1.x, x[1][s][1] - f1.y);
      ql[s][2] = pack_bf16x2(x[0][s][2] - f2.x, x[0][s][3] - f2.y);
      ql[s][3] = pack_bf16x2(x[1][s][2] - f3.x, x[1][s][3] - f3.y);
    }
  }

  float o[8][4];
#pragma unroll
  for (int d = 0; d < 8; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  int consumed = 0;  // pages whose copy this thread has seen land
  bool failed = false;

  for (int pg = 0; pg < n_pages; ++pg) {
    const int s = pg % C::kStages;
    const bool landed = mbar_wait_bounded(smem_addr(&full_bar[s]), (pg / C::kStages) & 1u);
    if (!__all_sync(kFull, landed)) {
      failed = true;
      break;
    }
    consumed = pg + 1;
    const int page = bt[pg];
    const bool bad = page < 0 || static_cast<long long>(page) >= p.num_pages;
    if (!bad) {
      const uint32_t sK = smem_addr(ring[s]), sV = sK + kHalfBytes;
      // S = Q K^T (16 rows x 16 keys; n-tiles j: keys 8j..8j+7), Q as hi and lo products
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
        for (int k = 0; k < 4; ++k) {
          mma_bf16_16816(sc[j], qh[k], kb[j][k][0], kb[j][k][1]);
          mma_bf16_16816(sc[j], ql[k], kb[j][k][0], kb[j][k][1]);
        }
      }
      // causal mask: key position key0 + 8j + 2tig (+1) must not pass the row's position
      const int key0 = pg * kPage;
      if (key0 + kPage - 1 > min(pos[0], pos[1])) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (key0 + 8 * j + 2 * tig + (c & 1) > pos[c >> 1]) sc[j][c] = -INFINITY;
      }
      // online softmax per row (row g8: c = 0, 1; row g8 + 8: c = 2, 3); page 0
      // holds key 0, which every row sees, so m_run is finite from then on
      float pr[2][4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float pm = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]), fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
        pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 1));
        pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 2));
        const float m_new = fmaxf(m_run[rr], pm);
        const float alpha = m_new > m_run[rr] ? fast_exp2(m_run[rr] - m_new) : 1.f;
        pr[rr][0] = fast_exp2(sc[0][2 * rr] - m_new);
        pr[rr][1] = fast_exp2(sc[0][2 * rr + 1] - m_new);
        pr[rr][2] = fast_exp2(sc[1][2 * rr] - m_new);
        pr[rr][3] = fast_exp2(sc[1][2 * rr + 1] - m_new);
        l_run[rr] = l_run[rr] * alpha + ((pr[rr][0] + pr[rr][1]) + (pr[rr][2] + pr[rr][3]));
        m_run[rr] = m_new;
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          o[d][2 * rr] *= alpha;
          o[d][2 * rr + 1] *= alpha;
        }
      }
      // P as the A operand (a0: row g8, keys 2tig..; a1: row g8+8; a2, a3: keys 8+2tig..),
      // once as bf16 and once as the bf16 remainder
      uint32_t ph[4], pl[4];
      {
        const float pa[4][2] = {{pr[0][0], pr[0][1]}, {pr[1][0], pr[1][1]},
                                {pr[0][2], pr[0][3]}, {pr[1][2], pr[1][3]}};
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          ph[a] = pack_bf16x2(pa[a][0], pa[a][1]);
          const float2 f = bf16x2_to_float2(ph[a]);
          pl[a] = pack_bf16x2(pa[a][0] - f.x, pa[a][1] - f.y);
        }
      }
      // O += P V (n-tiles d: dims 8d..8d+7), V fragments transposed by ldmatrix
      uint32_t vb[8][2];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int chunk = 2 * q + (mi >> 1), row = 8 * (mi & 1) + ri;
        ldsm_x4_trans(sV + row * kRowBytes + ((chunk ^ ri) << 4), vb[2 * q][0], vb[2 * q][1],
                      vb[2 * q + 1][0], vb[2 * q + 1][1]);
      }
      const int nv = last_pos - key0 + 1;  // slots holding keys of the tile
      if (nv < kPage) {  // later slots were never written: keep their bits out of P V
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
      for (int d = 0; d < 8; ++d) {
        mma_bf16_16816(o[d], ph, vb[d][0], vb[d][1]);
        mma_bf16_16816(o[d], pl, vb[d][0], vb[d][1]);
      }
    }
    // Release the stage. Thread 0 refills the stage of the previous page, one
    // page behind, so it rarely waits for the slower warps.
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
    if (warp == 0) {
      const int prev = pg - 1;
      bool ok = true;
      if (lane == 0 && prev >= 0 && prev + C::kStages < n_pages) {
        const int ps = prev % C::kStages;
        ok = mbar_wait_bounded(smem_addr(&empty_bar[ps]), (prev / C::kStages) & 1u);
        if (ok) issue(prev + C::kStages, ps);
      }
      if (!__shfl_sync(kFull, ok, 0)) {
        failed = true;
        break;
      }
    }
  }

  if (failed) {
    // Report; the issuing thread then lets every copy it started land before
    // the CTA's shared memory is released (a stage has one copy at a time).
    if (lane == 0) atomicOr(p.err, PKV_ERR_TIMEOUT);
    if (tid == 0) {
      for (int pg = consumed; pg < issued; ++pg)
        mbar_wait_bounded(smem_addr(&full_bar[pg % C::kStages]), (pg / C::kStages) & 1u);
    }
    return;
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    float l = l_run[rr] + __shfl_xor_sync(kFull, l_run[rr], 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (!live[rr]) continue;
    const int R = 16 * warp + g8 + 8 * rr;
    const int t = R / G, i = R - t * G;
    float* dst = p.out + (static_cast<size_t>(row0 + t) * p.hq + h * G + i) * kHeadDim;
    const float inv = 1.f / l;
#pragma unroll
    for (int d = 0; d < 8; ++d)
      *reinterpret_cast<float2*>(dst + 8 * d + 2 * tig) =
          make_float2(o[d][2 * rr] * inv, o[d][2 * rr + 1] * inv);
  }
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// Workspace: the expanded per-token tables, lengths and positions the append
// kernel reads, then the tile list and its count.
struct PrefillLayout {
  size_t tables, lens, pos, tiles, count, total;
};

// An upper bound on the tiles of any split of total_tokens over the batch
// (at most one partial tile per sequence); tokens per tile are at least 16.
size_t max_tiles(int total_tokens, int batch) {
  return static_cast<size_t>(total_tokens) / 16 + static_cast<size_t>(batch) + 1;
}

PrefillLayout layout(int total_tokens, int batch, int max_blocks) {
  PrefillLayout l;
  l.tables = 0;
  l.lens = l.tables + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens) * max_blocks);
  l.pos = l.lens + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens));
  l.tiles = l.pos + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens));
  l.count = l.tiles + align256(sizeof(int4) * max_tiles(total_tokens, batch));
  l.total = l.count + 256;
  return l;
}

template <int G>
cudaError_t launch_attn(const PrefillLaunch& a, const PrefillLayout& l, cudaStream_t stream) {
  using C = PrefillCfg<G>;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int4* tiles = reinterpret_cast<int4*>(ws + l.tiles);
  int* count = reinterpret_cast<int*>(ws + l.count);
  const size_t grid_x = static_cast<size_t>(a.total_tokens + C::kTokens - 1) / C::kTokens + a.batch;
  prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.cu_tokens, a.start_pos, a.batch,
                                                      a.total_tokens, C::kTokens,
                                                      static_cast<int>(grid_x), tiles, count, a.err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  PrefillAttnParams p;
  p.q_rot = a.q_rot;
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.max_blocks = a.max_blocks;
  p.tiles = tiles;
  p.num_tiles = count;
  p.hkv = a.num_kv_heads;
  p.hq = a.num_q_heads;
  p.num_pages = a.num_pages;
  p.qscale = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.err = a.err;
  const dim3 grid(static_cast<unsigned>(grid_x), static_cast<unsigned>(a.num_kv_heads));
  prefill_attn_kernel<G><<<grid, C::kThreads, 0, stream>>>(*a.kv_map, p);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_workspace_bytes(int total_tokens, int batch, int max_blocks) {
  return layout(total_tokens, batch, max_blocks).total;
}

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t stream) {
  if (a.total_tokens == 0) return cudaSuccess;
  const PrefillLayout l = layout(a.total_tokens, a.batch, a.max_blocks);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int32_t* tok_tables = reinterpret_cast<int32_t*>(ws + l.tables);
  int32_t* tok_lens = reinterpret_cast<int32_t*>(ws + l.lens);
  int32_t* tok_pos = reinterpret_cast<int32_t*>(ws + l.pos);
  prefill_expand_kernel<<<a.total_tokens, kExpandThreads, 0, stream>>>(
      a.block_tables, a.max_blocks, a.cu_tokens, a.start_pos, a.batch, a.total_tokens, tok_tables,
      tok_lens, tok_pos);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  AppendLaunch ap;
  ap.pool = const_cast<uint16_t*>(reinterpret_cast<const uint16_t*>(a.pool));
  ap.num_pages = a.num_pages;
  ap.num_kv_heads = a.num_kv_heads;
  ap.q = a.q;
  ap.k = a.k;
  ap.v = a.v;
  ap.q_rot = a.q_rot;
  ap.block_tables = tok_tables;
  ap.max_blocks = a.max_blocks;
  ap.seq_lens = tok_lens;
  ap.positions = tok_pos;
  ap.batch = a.total_tokens;
  ap.num_q_heads = a.num_q_heads;
  ap.rope_theta = a.rope_theta;
  ap.err = a.err;
  e = launch_append_rope(ap, stream);
  if (e != cudaSuccess) return e;

  switch (a.num_q_heads / a.num_kv_heads) {
    case 1: return launch_attn<1>(a, l, stream);
    case 2: return launch_attn<2>(a, l, stream);
    case 3: return launch_attn<3>(a, l, stream);
    case 4: return launch_attn<4>(a, l, stream);
    case 5: return launch_attn<5>(a, l, stream);
    case 6: return launch_attn<6>(a, l, stream);
    case 7: return launch_attn<7>(a, l, stream);
    case 8: return launch_attn<8>(a, l, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
