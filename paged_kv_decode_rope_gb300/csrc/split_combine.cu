// split_combine.cu -- log-sum-exp merge of split-KV partial results.
//
// Flash-decoding merge (not on the source pages; defined by its closed form):
// row r has num_splits[r] partial results (o_j normalised, lse_j the natural
// log-sum-exp of the split's scaled scores); with M = max_j lse_j and
// w_j = exp(lse_j - M) the merged row is sum_j w_j o_j / sum_j w_j.
// One warp per row. Lanes first take one split each (max, weights, their
// sum), then the lanes stride over head_dim and sum the weighted rows, the
// loads of different splits independent of each other.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCombineWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(kCombineWarps * 32)
    split_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                         const int32_t* __restrict__ num_splits, float* __restrict__ out, int rows,
                         int max_splits, int head_dim) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int ns = num_splits[row];
  float* o = out + static_cast<size_t>(row) * head_dim;
  const float* lse = lse_part + static_cast<size_t>(row) * max_splits;
  const float* op = o_part + static_cast<size_t>(row) * max_splits * head_dim;
  const bool valid = ns >= 1 && ns <= max_splits;
  float m = -INFINITY;
  if (valid)
    for (int j = lane; j < ns; j += 32) m = fmaxf(m, lse[j]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  if (!valid || m == -INFINITY || m != m) {  // bad count, empty or NaN row
    for (int d = lane; d < head_dim; d += 32) o[d] = 0.f;
    return;
  }
  float wsum = 0.f;
  for (int j = lane; j < ns; j += 32) wsum += exp2f((lse[j] - m) * kLog2e);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(kFull, wsum, off);
  const float inv = 1.f / wsum;
  for (int d0 = 0; d0 < head_dim; d0 += 32) {
    const int d = d0 + lane;
    float acc = 0.f;
    for (int j0 = 0; j0 < ns; j0 += 32) {
      const float wl = (j0 + lane < ns) ? exp2f((lse[j0 + lane] - m) * kLog2e) : 0.f;
      const int n = min(32, ns - j0);
#pragma unroll 8
      for (int t = 0; t < n; ++t) {
        const float w = __shfl_sync(kFull, wl, t);
        if (d < head_dim) acc += w * op[static_cast<size_t>(j0 + t) * head_dim + d];
      }
    }
    if (d < head_dim) o[d] = acc * inv;
  }
}

}  // namespace

cudaError_t launch_split_combine(const float* o_part, const float* lse_part,
                                 const int32_t* num_splits, float* out, int rows, int max_splits,
                                 int head_dim, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int grid = (rows + kCombineWarps - 1) / kCombineWarps;
  split_combine_kernel<<<grid, kCombineWarps * 32, 0, stream>>>(o_part, lse_part, num_splits, out,
                                                                rows, max_splits, head_dim);
  return cudaGetLastError();
}

}  // namespace pkv
