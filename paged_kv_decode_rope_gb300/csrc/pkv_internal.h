// pkv_internal.h -- host-side interfaces between the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

struct pkv_pool {
  // TMA descriptor of the pool seen as a 2-D bf16 tensor of 128-byte rows
  // (one token's K or V of one kv head): [num_pages*num_kv_heads*2*16][64],
  // 32-row boxes (a kv head's K and V rows of one page), 128-byte swizzle.
  CUtensorMap kv_map;  // 64-byte aligned by its type
  // the same tensor with 16-row boxes (a kv head's K rows, or V rows, of one page)
  CUtensorMap kv16_map;
  void* storage;
  size_t storage_bytes;
  long long num_pages;
  int num_kv_heads;
  int* d_err;  // device error word (PKV_ERR_* bits)
  int device;
  // looks a decode's merger takes at another CTA's partial before it gives
  // up with PKV_ERR_TIMEOUT (kv_pool_set_merge_wait_limit)
  uint32_t merge_looks;
};

namespace pkv {

constexpr int kMaxKvHeads = 256;
// Default bound of a merger's wait: looks at another CTA's partial, each an
// L2 round trip of about a microsecond, so a second or more where a partial
// comes within a few microseconds.
constexpr uint32_t kDefaultMergeLooks = 1u << 20;

struct AppendLaunch {
  uint16_t* pool;
  long long num_pages;
  int num_kv_heads;
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  float* q_rot;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* seq_lens;
  const int32_t* positions;
  int batch;
  int num_q_heads;
  double rope_theta;
  int* err;
};

cudaError_t launch_append_rope(const AppendLaunch& a, cudaStream_t stream);

struct DecodeLaunch {
  const CUtensorMap* kv_map;
  const uint8_t* pool;
  long long num_pages;
  int num_kv_heads;
  const float* q_rot;
  float* out;  // fused mode
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* seq_lens;
  int batch;
  int num_q_heads;
  float scale;
  int pages_per_split;  // 0 = balance over the persistent grid
  // fused merge: workspace (counters first, then partial slots)
  void* workspace;
  size_t workspace_bytes;
  // partials mode (o_part != nullptr)
  float* o_part;
  float* lse_part;
  int32_t* num_splits;
  int max_splits;
  int* err;
  uint32_t merge_looks;  // bound of a merger's wait for other CTAs' partials
  // the fused step (q_raw != nullptr): RoPE + append of the new token, then the decode
  const uint16_t* q_raw;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const void* rope_table;   // RoPE table of rope_positions rows, row p = position p
  int rope_positions;
  const int32_t* positions;  // [batch] RoPE position of each new token
  float* q_rot_out;
};

// Chunked causal prefill (prefill.cu): every chunk token becomes a one-token
// virtual sequence for the append and decode launches.
struct PrefillLaunch {
  const CUtensorMap* kv_map;
  const CUtensorMap* kv16_map;
  const uint8_t* pool;
  long long num_pages;
  int num_kv_heads;
  const uint16_t* q;  // bf16 [total_tokens][num_q_heads][64]
  const uint16_t* k;  // bf16 [total_tokens][num_kv_heads][64]
  const uint16_t* v;
  float* q_rot;       // fp32 [total_tokens][num_q_heads][64] out
  float* out;         // fp32 [total_tokens][num_q_heads][64] out
  const int32_t* block_tables;  // [batch][max_blocks]
  int max_blocks;
  const int32_t* cu_tokens;     // [batch + 1]
  const int32_t* start_pos;     // [batch]
  int batch;
  int total_tokens;
  int num_q_heads;
  float scale;
  const void* rope_table;  // RoPE table of rope_positions rows, row p = position p
  int rope_positions;
  void* workspace;
  size_t workspace_bytes;
  int sm_count;
  int* err;
};

size_t prefill_workspace_bytes(int total_tokens, int batch, int max_blocks);
cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t stream);

// Largest batch one decode launch serves (sequence lengths and page prefix sums
// are staged in shared memory); larger batches are cut into several launches.
constexpr int kDecodeBatchChunk = 2048;

size_t decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int max_blocks,
                              int pages_per_split, int sm_count);
cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t stream);
// The step's work plan in the decode workspace (positions null: for the
// decode from q_rot, whose lengths are not checked against positions).
cudaError_t launch_plan(const int32_t* seq_lens, const int32_t* positions, int rope_positions,
                        int batch, int num_q_heads, int num_kv_heads, int max_blocks,
                        void* workspace, cudaStream_t stream);

// cos and sin of pos * theta^(-2j/64), j < 32, for every row, correctly
// rounded to fp64, and split into fp32 pairs: table = float4 [rows][32]
// {cos_hi, cos_lo, sin_hi, sin_lo}, then double2 [rows][32] {cos, sin}
// (PKV_ROPE_TABLE_BYTES). Row r is position positions[r], or r when
// positions is null.
cudaError_t launch_rope_cos_sin(const int32_t* positions, int rows, double rope_theta,
                                void* table, cudaStream_t stream);

cudaError_t launch_split_combine(const float* o_part, const float* lse_part,
                                 const int32_t* num_splits, float* out, int rows, int max_splits,
                                 int head_dim, cudaStream_t stream);

int device_sm_count(int device);

// Remember a CUDA failure for pkv_last_cuda_error() (calling thread).
void record_cuda_error(cudaError_t e);

// Encode a TMA descriptor of the pool (see pkv_pool::kv_map) with boxes of
// box_rows rows.
cudaError_t encode_kv_map(CUtensorMap* map, void* storage, long long num_pages, int num_kv_heads,
                          int box_rows);

}  // namespace pkv
