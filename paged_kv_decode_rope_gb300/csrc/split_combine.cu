// split_combine.cu -- log-sum-exp merge of split-KV partial results.
//
// Flash-decoding merge (not on the source pages; defined by its closed form):
// row r has num_splits[r] partial results (o_j normalised, lse_j the natural
// log-sum-exp of the split's scaled scores); with M = max_j lse_j and
// w_j = exp(lse_j - M) the merged row is sum_j w_j o_j / sum_j w_j.
// One warp per row; lanes stride over head_dim. Tiny next to the decode
// (rows * splits * head_dim * 4 bytes).
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
  float m = -INFINITY;
  if (ns >= 1 && ns <= max_splits)
    for (int j = 0; j < ns; ++j) m = fmaxf(m, lse[j]);
  if (m == -INFINITY || m != m) {  // bad count, empty or NaN row
    for (int d = lane; d < head_dim; d += 32) o[d] = 0.f;
    return;
  }
  float wsum = 0.f;
  for (int j = 0; j < ns; ++j) wsum += exp2f((lse[j] - m) * kLog2e);
  const float inv = 1.f / wsum;
  for (int d = lane; d < head_dim; d += 32) {
    float acc = 0.f;
    for (int j = 0; j < ns; ++j) {
      const float w = exp2f((lse[j] - m) * kLog2e);
      acc += w * o_part[(static_cast<size_t>(row) * max_splits + j) * head_dim + d];
    }
    o[d] = acc * inv;
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
