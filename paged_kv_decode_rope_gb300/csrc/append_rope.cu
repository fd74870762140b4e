// append_rope.cu -- RoPE of the new token's q and k, and its append into the
// BF16 page pool.
//
// "Hours of YouTube and 85 handtyped pages of notes on LLM Inference – Start
// here", shared BF16 KV page pool item: decode writes one new token per
// sequence at its absolute RoPE position into the page its block table maps.
// "手写LLM推理引擎：Tokenizer、Transformer与Detokenizer三段式实现" section 3.2:
// the rotation y_j = x_j cos(m theta_j) - x_{j'} sin(m theta_j),
// y_{j'} = x_{j'} cos + x_j sin with theta_j = base^(-2j/D), read with
// rotate-half pairing j' = j + D/2.
//
// One CTA per sequence. 32 threads evaluate the 32 angles' cos/sin in fp64;
// the key is rotated in fp64 with explicitly rounded products and sums (no
// contraction) and rounded once to bf16, so the stored bytes are reproducible
// bit for bit. The query is rotated in fp32 and kept in fp32. Values are
// copied verbatim. The whole kernel moves B*(Hq+2*Hkv)*128 bytes: it is
// launch-latency bound, not bandwidth bound.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;
constexpr int kHalf = kHeadDim / 2;

struct InvFreq {
  double v[kHalf];  // theta^(-2j/64), evaluated on the host with the C library's pow
};

struct AppendParams {
  uint16_t* pool;
  long long num_pages;
  int hkv;
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  float* q_rot;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* seq_lens;
  const int32_t* positions;
  int hq;
  int* err;
  double inv_freq[kHalf];
};

__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(const AppendParams p) {
  __shared__ double cos_d[kHalf], sin_d[kHalf];
  __shared__ float cos_f[kHalf], sin_f[kHalf];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = p.seq_lens[b];
  const int pos = p.positions[b];
  if (tid < kHalf) {
    const double angle = __dmul_rn(static_cast<double>(pos), p.inv_freq[tid]);
    double s, c;
    sincos(angle, &s, &c);
    cos_d[tid] = c;
    sin_d[tid] = s;
    cos_f[tid] = static_cast<float>(c);
    sin_f[tid] = static_cast<float>(s);
  }
  __syncthreads();

  // Rotated query, fp32, [Hq][64].
  const uint16_t* qb = p.q + static_cast<size_t>(b) * p.hq * kHeadDim;
  float* qo = p.q_rot + static_cast<size_t>(b) * p.hq * kHeadDim;
  for (int idx = tid; idx < p.hq * kHalf; idx += kAppendThreads) {
    const int head = idx / kHalf, j = idx % kHalf;
    const float x0 = __uint_as_float(static_cast<uint32_t>(qb[head * kHeadDim + j]) << 16);
    const float x1 = __uint_as_float(static_cast<uint32_t>(qb[head * kHeadDim + j + kHalf]) << 16);
    qo[head * kHeadDim + j] = x0 * cos_f[j] - x1 * sin_f[j];
    qo[head * kHeadDim + j + kHalf] = x1 * cos_f[j] + x0 * sin_f[j];
  }

  // Destination slot of the new token.
  const int t = n - 1;
  bool ok = n >= 1 && n <= p.max_blocks * kPage;
  long long page = -1;
  if (ok) {
    page = p.block_tables[static_cast<size_t>(b) * p.max_blocks + t / kPage];
    ok = page >= 0 && page < p.num_pages;
    if (!ok && tid == 0) atomicOr(p.err, PKV_ERR_PAGE_ID);
  } else if (tid == 0) {
    atomicOr(p.err, PKV_ERR_SEQ_LEN);
  }
  if (!ok) return;
  const int slot = t % kPage;
  uint16_t* page_base = p.pool + static_cast<size_t>(page) * p.hkv * (kHeadPageBytes / 2);

  // Rotated key: fp64, explicit roundings, one rounding to bf16.
  const uint16_t* kb = p.k + static_cast<size_t>(b) * p.hkv * kHeadDim;
  for (int idx = tid; idx < p.hkv * kHalf; idx += kAppendThreads) {
    const int h = idx / kHalf, j = idx % kHalf;
    uint16_t y0, y1;
    rotate_key_pair(kb[h * kHeadDim + j], kb[h * kHeadDim + j + kHalf], cos_d[j], sin_d[j], y0, y1);
    uint16_t* krow = page_base + (h * 2 + 0) * (kHalfBytes / 2) + slot * kHeadDim;
    krow[j] = y0;
    krow[j + kHalf] = y1;
  }
  // Value: 16-byte copies.
  const uint4* vb = reinterpret_cast<const uint4*>(p.v + static_cast<size_t>(b) * p.hkv * kHeadDim);
  for (int idx = tid; idx < p.hkv * (kRowBytes / 16); idx += kAppendThreads) {
    const int h = idx / (kRowBytes / 16), c = idx % (kRowBytes / 16);
    uint4* vrow = reinterpret_cast<uint4*>(page_base + (h * 2 + 1) * (kHalfBytes / 2) + slot * kHeadDim);
    vrow[c] = vb[h * (kRowBytes / 16) + c];
  }
}

// One thread per (sequence, frequency): cos and sin of pos * inv_freq_j in
// fp64 (the values the append kernel forms for its rotation), stored twice:
// as fp32 pairs {hi, lo} (hi = the fp64 value rounded to fp32, lo = the
// remainder rounded to fp32, so hi + lo is within 2^-48 of it) for the fused
// step's fp32 paths, and in fp64 for its rare fp64 fallback.
__global__ void rope_cos_sin_kernel(const int32_t* __restrict__ positions, int batch,
                                    const InvFreq inv, float4* __restrict__ pairs,
                                    double2* __restrict__ full) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= batch * kHalf) return;
  const int b = idx / kHalf, j = idx % kHalf;
  const double angle = __dmul_rn(static_cast<double>(positions[b]), inv.v[j]);
  double s, c;
  sincos(angle, &s, &c);
  const float ch = __double2float_rn(c), sh = __double2float_rn(s);
  pairs[idx] = make_float4(ch, __double2float_rn(__dsub_rn(c, static_cast<double>(ch))), sh,
                           __double2float_rn(__dsub_rn(s, static_cast<double>(sh))));
  full[idx] = make_double2(c, s);
}

}  // namespace

cudaError_t launch_rope_cos_sin(const int32_t* positions, int batch, double rope_theta,
                                void* table, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  InvFreq inv;
  for (int j = 0; j < kHalf; ++j)
    inv.v[j] = std::pow(rope_theta, -(2.0 * j) / static_cast<double>(kHeadDim));
  const int n = batch * kHalf;
  float4* pairs = static_cast<float4*>(table);
  double2* full = reinterpret_cast<double2*>(pairs + n);
  rope_cos_sin_kernel<<<(n + 255) / 256, 256, 0, stream>>>(positions, batch, inv, pairs, full);
  return cudaGetLastError();
}

cudaError_t launch_append_rope(const AppendLaunch& a, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  AppendParams p;
  p.pool = a.pool;
  p.num_pages = a.num_pages;
  p.hkv = a.num_kv_heads;
  p.q = a.q;
  p.k = a.k;
  p.v = a.v;
  p.q_rot = a.q_rot;
  p.block_tables = a.block_tables;
  p.max_blocks = a.max_blocks;
  p.seq_lens = a.seq_lens;
  p.positions = a.positions;
  p.hq = a.num_q_heads;
  p.err = a.err;
  // Step 1 of the rotation, the 32 inverse frequencies base^(-2j/64), is a
  // launch constant: it is evaluated once here with the C library's pow and
  // passed by value; each kernel thread then forms its angle pos * inv_freq_j
  // (one rounded product) and its cos/sin in fp64.
  for (int j = 0; j < kHalf; ++j)
    p.inv_freq[j] = std::pow(a.rope_theta, -(2.0 * j) / static_cast<double>(kHeadDim));
  append_rope_kernel<<<a.batch, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
