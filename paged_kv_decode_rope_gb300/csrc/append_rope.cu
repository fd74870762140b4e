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
// One CTA per sequence. 64 threads evaluate the 32 angles' cos and sin,
// correctly rounded to fp64 (rope_cr.cuh). The key is rotated and rounded to
// bf16 exactly as fp64 arithmetic on those values rounds it (two rounded
// products, one rounded difference, then one rounding to bf16): by the
// certified fp32 double-word path the fused decode step uses, with the fp64
// rotation where that path cannot certify, so the stored bytes are the same
// bit for bit whichever entry point appends. The query is rotated in fp32 and
// kept in fp32. Values are copied verbatim. The whole kernel moves
// B*(Hq+2*Hkv)*128 bytes: it is launch-latency bound, not bandwidth bound.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "rope_cr.cuh"

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
  RopeSeriesCoef coef;
};

__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(const AppendParams p) {
  __shared__ double cs_d[kHalf][2];  // {cos, sin}, correctly rounded fp64
  __shared__ float cs_f[kHalf][4];   // {cos_hi, cos_lo, sin_hi, sin_lo}
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = p.seq_lens[b];
  const int pos = p.positions[b];
  if (tid < 2 * kHalf) {  // thread 2j: cos of angle j, 2j + 1: its sin
    const int j = tid >> 1, w = tid & 1;
    bool certain;
    const double val = rope_cos_or_sin_cr(__dmul_rn(static_cast<double>(pos), p.inv_freq[j]), w != 0,
                                          p.coef, &certain);
    const float hi = __double2float_rn(val);
    cs_d[j][w] = val;
    cs_f[j][2 * w] = hi;
    cs_f[j][2 * w + 1] = __double2float_rn(__dsub_rn(val, static_cast<double>(hi)));
  }
  __syncthreads();

  // Rotated query, fp32, [Hq][64], from the fp32 roundings of cos and sin.
  const uint16_t* qb = p.q + static_cast<size_t>(b) * p.hq * kHeadDim;
  float* qo = p.q_rot + static_cast<size_t>(b) * p.hq * kHeadDim;
  for (int idx = tid; idx < p.hq * kHalf; idx += kAppendThreads) {
    const int head = idx / kHalf, j = idx % kHalf;
    const float x0 = __uint_as_float(static_cast<uint32_t>(qb[head * kHeadDim + j]) << 16);
    const float x1 = __uint_as_float(static_cast<uint32_t>(qb[head * kHeadDim + j + kHalf]) << 16);
    qo[head * kHeadDim + j] = x0 * cs_f[j][0] - x1 * cs_f[j][2];
    qo[head * kHeadDim + j + kHalf] = x1 * cs_f[j][0] + x0 * cs_f[j][2];
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

  // Rotated key, rounded once to bf16 as the fp64 rotation rounds it.
  const uint16_t* kb = p.k + static_cast<size_t>(b) * p.hkv * kHeadDim;
  for (int idx = tid; idx < p.hkv * kHalf; idx += kAppendThreads) {
    const int h = idx / kHalf, j = idx % kHalf;
    const uint16_t k0 = kb[h * kHeadDim + j], k1 = kb[h * kHeadDim + j + kHalf];
    const float x0 = __uint_as_float(static_cast<uint32_t>(k0) << 16);
    const float x1 = __uint_as_float(static_cast<uint32_t>(k1) << 16);
    const float* c = cs_f[j];
    uint16_t y0, y1;
    if (!(rotated_bf16_fast(x0, x1, c[0], c[1], c[2], c[3], y0) &&
          rotated_bf16_fast(x1, -x0, c[0], c[1], c[2], c[3], y1)))
      rotate_key_pair(k0, k1, cs_d[j][0], cs_d[j][1], y0, y1);
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

// Two threads per (row, frequency), one for the cos and one for the sin of
// pos * inv_freq_j (pos = positions[row], or the row itself), correctly
// rounded to fp64 (the values the append kernel forms for its rotation),
// stored twice: as fp32 pairs {hi, lo} (hi = the fp64 value rounded to fp32,
// lo = the remainder rounded to fp32, so hi + lo is within 2^-48 of it) for
// the fp32 paths of the fused step and the prefill, and in fp64 for their
// rare fp64 fallback. Small blocks spread the values over as many SMs as the
// rows allow: each value is a long chain of dependent fp64 operations.
constexpr int kTableThreads = 64;
__global__ void __launch_bounds__(kTableThreads)
    rope_cos_sin_kernel(const int32_t* __restrict__ positions, int batch, const InvFreq inv,
                        const RopeSeriesCoef coef, float2* __restrict__ pairs,
                        double* __restrict__ full) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;  // 2 (b 32 + j) + (0: cos, 1: sin)
  if (idx >= batch * 2 * kHalf) return;
  const int bj = idx >> 1, b = bj / kHalf, j = bj - b * kHalf;
  const int pos = positions ? positions[b] : b;
  bool certain;
  const double val = rope_cos_or_sin_cr(__dmul_rn(static_cast<double>(pos), inv.v[j]),
                                        (idx & 1) != 0, coef, &certain);
  const float hi = __double2float_rn(val);
  pairs[idx] = make_float2(hi, __double2float_rn(__dsub_rn(val, static_cast<double>(hi))));
  full[idx] = val;
}

}  // namespace

RopeSeriesCoef rope_series_coef() {
  RopeSeriesCoef c;
  for (int n = 0; n < 16; ++n) {
    // n = 0 is unused; 1/((2n-1)(2n)) and 1/((2n)(2n+1)) for n >= 1
    const double dc = n ? static_cast<double>((2 * n - 1) * (2 * n)) : 1.0;
    const double ds = n ? static_cast<double>((2 * n) * (2 * n + 1)) : 1.0;
    c.cos_hi[n] = 1.0 / dc;
    c.cos_lo[n] = std::fma(-c.cos_hi[n], dc, 1.0) / dc;
    c.sin_hi[n] = 1.0 / ds;
    c.sin_lo[n] = std::fma(-c.sin_hi[n], ds, 1.0) / ds;
  }
  return c;
}

cudaError_t launch_rope_cos_sin(const int32_t* positions, int batch, double rope_theta,
                                void* table, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  if (static_cast<long long>(batch) * 2 * kHalf >= (1ll << 31)) return cudaErrorInvalidValue;
  InvFreq inv;
  for (int j = 0; j < kHalf; ++j)
    inv.v[j] = std::pow(rope_theta, -(2.0 * j) / static_cast<double>(kHeadDim));
  const int n = batch * 2 * kHalf;
  float2* pairs = static_cast<float2*>(table);
  double* full = reinterpret_cast<double*>(pairs + n);
  rope_cos_sin_kernel<<<(n + kTableThreads - 1) / kTableThreads, kTableThreads, 0, stream>>>(
      positions, batch, inv, rope_series_coef(), pairs, full);
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
  // (one rounded product) and its correctly rounded fp64 cos or sin.
  for (int j = 0; j < kHalf; ++j)
    p.inv_freq[j] = std::pow(a.rope_theta, -(2.0 * j) / static_cast<double>(kHeadDim));
  p.coef = rope_series_coef();
  append_rope_kernel<<<a.batch, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
