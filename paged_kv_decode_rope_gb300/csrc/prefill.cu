// prefill.cu -- chunked causal prefill into the page pool.
//
// "Hours of YouTube and 85 handtyped pages of notes on LLM Inference – Start
// here": prefill fills the prompt pages (dense causal prefill), decode then
// appends one token at a time. A chunk of new tokens for sequence b sits at
// positions start_pos[b], start_pos[b]+1, ...; every chunk token is rotated
// and appended like a decode token, and the queries of chunk token t attend
// causally over the sequence's first start_pos[b] + t + 1 tokens.
//
// Built on the decode path: each chunk token becomes a one-token "virtual
// sequence" with its own length (its causal prefix) and its sequence's block
// table row. One small kernel expands those rows; the append kernel then
// rotates and stores every chunk token, and the decode kernel (with its
// split-KV merge) attends for every token. The prefix pages a chunk's tokens
// share are read once per token, mostly from L2 (a chunk's pages are small
// next to L2); a dedicated prefill kernel with query tiles would read them
// once per tile.
#include <cerrno>

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

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

struct PrefillLayout {
  size_t tables, lens, pos, decode, total;
};

PrefillLayout layout(int total_tokens, int num_q_heads, int num_kv_heads, int max_blocks,
                     int sm_count) {
  PrefillLayout l;
  l.tables = 0;
  l.lens = l.tables + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens) * max_blocks);
  l.pos = l.lens + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens));
  l.decode = l.pos + align256(sizeof(int32_t) * static_cast<size_t>(total_tokens));
  const size_t dec = decode_workspace_bytes(total_tokens, num_q_heads, num_kv_heads, max_blocks, 0,
                                            sm_count);
  l.total = dec == 0 ? 0 : l.decode + dec;
  return l;
}

}  // namespace

size_t prefill_workspace_bytes(int total_tokens, int num_q_heads, int num_kv_heads,
                               int max_blocks, int sm_count) {
  return layout(total_tokens, num_q_heads, num_kv_heads, max_blocks, sm_count).total;
}

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t stream) {
  if (a.total_tokens == 0) return cudaSuccess;
  const PrefillLayout l = layout(a.total_tokens, a.num_q_heads, a.num_kv_heads, a.max_blocks,
                                 a.sm_count);
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

  DecodeLaunch d = {};
  d.kv_map = a.kv_map;
  d.pool = a.pool;
  d.num_pages = a.num_pages;
  d.num_kv_heads = a.num_kv_heads;
  d.q_rot = a.q_rot;
  d.out = a.out;
  d.block_tables = tok_tables;
  d.max_blocks = a.max_blocks;
  d.seq_lens = tok_lens;
  d.batch = a.total_tokens;
  d.num_q_heads = a.num_q_heads;
  d.scale = a.scale;
  d.pages_per_split = 0;
  d.workspace = ws + l.decode;
  d.workspace_bytes = l.total - l.decode;
  d.err = a.err;
  return launch_decode(d, stream);
}

}  // namespace pkv
