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

__device__ __forceinline__ double bf16_bits_to_double(uint16_t b) {
  return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
}

// Round a double to the nearest bf16, ties to even, by integer manipulation
// of its IEEE-754 encoding. NaN becomes the quiet NaN 0x7FC0.
__device__ __forceinline__ uint16_t double_to_bf16_rne(double x) {
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  const uint16_t sign = static_cast<uint16_t>((u >> 48) & 0x8000u);
  const int biased = static_cast<int>((u >> 52) & 0x7ff);
  const unsigned long long frac = u & ((1ull << 52) - 1);
  if (biased == 0x7ff) return frac ? 0x7FC0 : static_cast<uint16_t>(sign | 0x7F80);
  if (biased == 0) return sign;  // |x| < 2^-1022 rounds to zero in bf16
  int e = biased - 1023;
  const unsigned long long sig = frac | (1ull << 52);  // 53-bit significand
  // bits to drop: to 8 significant bits for a normal bf16, more below 2^-126
  const int shift = (e >= -126) ? 45 : 45 + (-126 - e);
  if (shift >= 64) return sign;
  unsigned long long kept = sig >> shift;
  const unsigned long long rem = sig & ((1ull << shift) - 1);
  const unsigned long long half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (kept & 1))) ++kept;
  if (e >= -126) {
    if (kept == (1ull << 8)) {  // carried into the next binade
      kept >>= 1;
      ++e;
    }
    if (e > 127) return static_cast<uint16_t>(sign | 0x7F80);
    return static_cast<uint16_t>(sign | ((e + 127) << 7) | (kept & 0x7f));
  }
  // subnormal bf16 (kept <= 128; 128 is the smallest normal, encoded the same way)
  return static_cast<uint16_t>(sign | kept);
}

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
    const double x0 = bf16_bits_to_double(kb[h * kHeadDim + j]);
    const double x1 = bf16_bits_to_double(kb[h * kHeadDim + j + kHalf]);
    const double c = cos_d[j], s = sin_d[j];
    const double y0 = __dsub_rn(__dmul_rn(x0, c), __dmul_rn(x1, s));
    const double y1 = __dadd_rn(__dmul_rn(x1, c), __dmul_rn(x0, s));
    uint16_t* krow = page_base + (h * 2 + 0) * (kHalfBytes / 2) + slot * kHeadDim;
    krow[j] = double_to_bf16_rne(y0);
    krow[j + kHalf] = double_to_bf16_rne(y1);
  }
  // Value: 16-byte copies.
  const uint4* vb = reinterpret_cast<const uint4*>(p.v + static_cast<size_t>(b) * p.hkv * kHeadDim);
  for (int idx = tid; idx < p.hkv * (kRowBytes / 16); idx += kAppendThreads) {
    const int h = idx / (kRowBytes / 16), c = idx % (kRowBytes / 16);
    uint4* vrow = reinterpret_cast<uint4*>(page_base + (h * 2 + 1) * (kHalfBytes / 2) + slot * kHeadDim);
    vrow[c] = vb[h * (kRowBytes / 16) + c];
  }
}

}  // namespace

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
