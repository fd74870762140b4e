// pkv_abi.cu -- the C ABI declared in include/pkv.h: argument checks, the pool
// handle, and the launches. Returns 0 or a negative errno, the convention of
// "llmc — 从零写一个大模型推理引擎（配套代码）" (introduction).
#include <cerrno>
#include <cmath>
#include <cstdlib>
#include <new>

#include <cudaTypedefs.h>

#include "../../include/pkv.h"
#include "pkv_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return -EIO;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool geometry_ok(int num_kv_heads, int head_dim, int page_size) {
  return num_kv_heads >= 1 && num_kv_heads <= pkv::kMaxKvHeads && head_dim == PKV_HEAD_DIM &&
         page_size == PKV_PAGE_SIZE;
}

// Shapes shared by the decode entry points.
bool decode_shape_ok(const pkv_pool_t* pool, int batch, int num_q_heads, int max_blocks) {
  if (!pool || batch < 0 || max_blocks < 1 || num_q_heads < 1) return false;
  if (num_q_heads % pool->num_kv_heads) return false;
  const int group = num_q_heads / pool->num_kv_heads;
  if (group > PKV_MAX_GROUP) return false;
  // work items (sequence, kv head, page) of one launch are counted in int32
  const long long chunk = batch < pkv::kDecodeBatchChunk ? batch : pkv::kDecodeBatchChunk;
  if (chunk * pool->num_kv_heads * max_blocks >= (1ll << 31)) return false;
  if (static_cast<long long>(max_blocks) * PKV_PAGE_SIZE >= (1ll << 31)) return false;
  return true;
}

}  // namespace

namespace pkv {

cudaError_t encode_kv_map(CUtensorMap* map, void* storage, long long num_pages, int num_kv_heads,
                          int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // rows of 64 bf16 (128 B): one token's K or V of one kv head, row index
  // ((page * num_kv_heads + h) * 2 + kind) * 16 + slot
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(PKV_HEAD_DIM),
                              static_cast<cuuint64_t>(num_pages) * num_kv_heads * 2 * PKV_PAGE_SIZE};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(PKV_HEAD_DIM) * 2};
  // a box of 32 rows = one kv head's K and V rows of one page (4 KiB); of 16
  // rows = its K rows or its V rows
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(PKV_HEAD_DIM), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, storage, dims, strides, box, elem,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

int device_sm_count(int device) {
  static int cache[64] = {0};
  const int d = device & 63;
  if (cache[d] > 0) return cache[d];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -1;
  cache[d] = n;
  return n;
}
}  // namespace pkv

extern "C" {

size_t kv_pool_page_bytes(int num_kv_heads, int head_dim, int page_size) {
  if (!geometry_ok(num_kv_heads, head_dim, page_size)) return 0;
  return static_cast<size_t>(num_kv_heads) * 2 * page_size * head_dim * 2;
}

int kv_pool_create(pkv_pool_t** pool, void* storage, size_t storage_bytes, int num_kv_heads,
                   int head_dim, int page_size) {
  if (!pool) return -EINVAL;
  *pool = nullptr;
  if (!storage || !aligned16(storage) || !geometry_ok(num_kv_heads, head_dim, page_size))
    return -EINVAL;
  const size_t page_bytes = kv_pool_page_bytes(num_kv_heads, head_dim, page_size);
  const size_t pages = storage_bytes / page_bytes;
  if (pages == 0) return -ENOSPC;
  // token rows (page, head, K/V, slot) are addressed with 32-bit coordinates
  if (pages * static_cast<size_t>(num_kv_heads) * 2 * page_size >= (1ull << 31)) return -EINVAL;
  pkv_pool_t* h = new (std::nothrow) pkv_pool_t;
  if (!h) return -ENOMEM;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e == cudaSuccess)
    e = pkv::encode_kv_map(&h->kv_map, storage, static_cast<long long>(pages), num_kv_heads, 2 * page_size);
  if (e == cudaSuccess)
    e = pkv::encode_kv_map(&h->kv16_map, storage, static_cast<long long>(pages), num_kv_heads, page_size);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e);
  }
  int* d_err = nullptr;
  e = cudaMalloc(&d_err, sizeof(int));
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e);
  }
  e = cudaMemset(d_err, 0, sizeof(int));
  if (e != cudaSuccess) {
    cudaFree(d_err);
    delete h;
    return cuda_fail(e);
  }
  h->storage = storage;
  h->storage_bytes = storage_bytes;
  h->num_pages = static_cast<long long>(pages);
  h->num_kv_heads = num_kv_heads;
  h->d_err = d_err;
  h->device = device;
  h->merge_looks = pkv::kDefaultMergeLooks;
  *pool = h;
  return 0;
}

int kv_pool_destroy(pkv_pool_t* pool) {
  if (!pool) return 0;
  cudaError_t e = cudaFree(pool->d_err);
  delete pool;
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int kv_pool_num_pages(const pkv_pool_t* pool) {
  if (!pool) return -EINVAL;
  return static_cast<int>(pool->num_pages);
}

int kv_pool_set_merge_wait_limit(pkv_pool_t* pool, uint32_t looks, uint32_t* previous) {
  if (!pool) return -EINVAL;
  if (previous) *previous = pool->merge_looks;
  pool->merge_looks = looks;
  return 0;
}

int paged_kv_append_rope(pkv_pool_t* pool, const void* q, const void* k, const void* v,
                         float* q_rot, const int32_t* block_tables, int max_blocks,
                         const int32_t* seq_lens, const int32_t* positions, int batch,
                         int num_q_heads, double rope_theta, void* stream) {
  if (!pool || batch < 0 || max_blocks < 1 || num_q_heads < 1 ||
      num_q_heads % pool->num_kv_heads || !(rope_theta > 0.0) || !std::isfinite(rope_theta))
    return -EINVAL;
  if (static_cast<long long>(max_blocks) * PKV_PAGE_SIZE >= (1ll << 31)) return -EINVAL;
  if (batch == 0) return 0;
  if (!q || !k || !v || !q_rot || !block_tables || !seq_lens || !positions) return -EINVAL;
  if (!aligned16(v)) return -EINVAL;
  pkv::AppendLaunch a;
  a.pool = static_cast<uint16_t*>(pool->storage);
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.q_rot = q_rot;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.positions = positions;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.rope_theta = rope_theta;
  a.err = pool->d_err;
  cudaError_t e = pkv::launch_append_rope(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

size_t paged_gqa_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                        int max_blocks, int pages_per_split) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return 0;
  const int sms = pkv::device_sm_count(device);
  if (sms < 1) return 0;
  return pkv::decode_workspace_bytes(batch, num_q_heads, num_kv_heads, max_blocks, pages_per_split,
                                     sms);
}

int paged_gqa_decode(const pkv_pool_t* pool, const float* q_rot, float* out,
                     const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                     int batch, int num_q_heads, float scale, int pages_per_split,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!decode_shape_ok(pool, batch, num_q_heads, max_blocks) || pages_per_split < 0 ||
      !std::isfinite(scale))
    return -EINVAL;
  if (batch == 0) return 0;
  if (!q_rot || !out || !block_tables || !seq_lens || !workspace) return -EINVAL;
  if (!aligned16(q_rot) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return -EINVAL;
  const size_t need = paged_gqa_decode_workspace_bytes(batch, num_q_heads, pool->num_kv_heads,
                                                       max_blocks, pages_per_split);
  if (need == 0 || workspace_bytes < need) return -EINVAL;
  pkv::DecodeLaunch a = {};
  a.kv_map = &pool->kv_map;
  a.pool = static_cast<const uint8_t*>(pool->storage);
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.q_rot = q_rot;
  a.out = out;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.pages_per_split = pages_per_split;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err = pool->d_err;
  a.merge_looks = pool->merge_looks;
  cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int paged_decode_plan(const pkv_pool_t* pool, const int32_t* seq_lens, const int32_t* positions,
                      int rope_positions, int batch, int num_q_heads, int max_blocks,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!decode_shape_ok(pool, batch, num_q_heads, max_blocks)) return -EINVAL;
  if (positions && (rope_positions < 1 || rope_positions >= (1 << 24))) return -EINVAL;
  if (batch == 0 || batch > pkv::kDecodeBatchChunk) return 0;  // nothing to plan
  if (!seq_lens || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return -EINVAL;
  const size_t need = paged_gqa_decode_workspace_bytes(batch, num_q_heads, pool->num_kv_heads,
                                                       max_blocks, 0);
  if (need == 0 || workspace_bytes < need) return -EINVAL;
  cudaError_t e = pkv::launch_plan(seq_lens, positions, rope_positions, batch, num_q_heads,
                                   pool->num_kv_heads, max_blocks, workspace,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int paged_rope_cos_sin(const int32_t* positions, int rows, double rope_theta, void* table,
                       void* stream) {
  if (rows < 0 || rows >= (1 << 24) || !(rope_theta > 0.0) || !std::isfinite(rope_theta))
    return -EINVAL;
  if (rows == 0) return 0;
  if (!positions || !table || !aligned16(table)) return -EINVAL;
  cudaError_t e = pkv::launch_rope_cos_sin(positions, rows, rope_theta, table,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int paged_rope_table_build(double rope_theta, int num_positions, void* table, void* stream) {
  if (num_positions < 1 || num_positions >= (1 << 24) || !(rope_theta > 0.0) ||
      !std::isfinite(rope_theta))
    return -EINVAL;
  if (!table || !aligned16(table)) return -EINVAL;
  cudaError_t e = pkv::launch_rope_cos_sin(nullptr, num_positions, rope_theta, table,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int paged_decode_step(pkv_pool_t* pool, const void* q, const void* k, const void* v,
                      const void* rope_table, int rope_positions, const int32_t* positions,
                      float* q_rot, float* out, const int32_t* block_tables, int max_blocks,
                      const int32_t* seq_lens, int batch, int num_q_heads, float scale,
                      int pages_per_split, void* workspace, size_t workspace_bytes, void* stream) {
  if (!decode_shape_ok(pool, batch, num_q_heads, max_blocks) || pages_per_split < 0 ||
      !std::isfinite(scale) || rope_positions < 1 || rope_positions >= (1 << 24))
    return -EINVAL;
  if (batch == 0) return 0;
  if (!q || !k || !v || !rope_table || !positions || !out || !block_tables || !seq_lens ||
      !workspace)
    return -EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(rope_table) || !aligned16(out) ||
      (q_rot && !aligned16(q_rot)) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return -EINVAL;
  const size_t need = paged_gqa_decode_workspace_bytes(batch, num_q_heads, pool->num_kv_heads,
                                                       max_blocks, pages_per_split);
  if (need == 0 || workspace_bytes < need) return -EINVAL;
  pkv::DecodeLaunch a = {};
  a.kv_map = &pool->kv_map;
  a.pool = static_cast<const uint8_t*>(pool->storage);
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.out = out;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.pages_per_split = pages_per_split;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err = pool->d_err;
  a.q_raw = static_cast<const uint16_t*>(q);
  a.k_new = static_cast<const uint16_t*>(k);
  a.v_new = static_cast<const uint16_t*>(v);
  a.rope_table = rope_table;
  a.rope_positions = rope_positions;
  a.positions = positions;
  a.q_rot_out = q_rot;
  a.merge_looks = pool->merge_looks;
  cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

size_t paged_prefill_workspace_bytes(int total_tokens, int batch, int max_blocks) {
  if (total_tokens < 0 || batch < 1 || max_blocks < 1) return 0;
  return pkv::prefill_workspace_bytes(total_tokens, batch, max_blocks);
}

int paged_prefill(pkv_pool_t* pool, const void* q, const void* k, const void* v, float* q_rot,
                  float* out, const int32_t* block_tables, int max_blocks,
                  const int32_t* cu_tokens, const int32_t* start_pos, int batch, int total_tokens,
                  int num_q_heads, const void* rope_table, int rope_positions, float scale,
                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!decode_shape_ok(pool, total_tokens, num_q_heads, max_blocks) || batch < 0 ||
      total_tokens < 0 || !std::isfinite(scale) || rope_positions < 1 ||
      rope_positions >= (1 << 24))
    return -EINVAL;
  if (total_tokens == 0) return 0;
  if (batch < 1) return -EINVAL;
  if (!q || !k || !v || !q_rot || !out || !block_tables || !cu_tokens || !start_pos ||
      !rope_table || !workspace)
    return -EINVAL;
  if (!aligned16(q) || !aligned16(q_rot) || !aligned16(out) || !aligned16(v) || !aligned16(rope_table) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return -EINVAL;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e);
  const int sms = pkv::device_sm_count(device);
  const size_t need = paged_prefill_workspace_bytes(total_tokens, batch, max_blocks);
  if (sms < 1 || need == 0 || workspace_bytes < need) return -EINVAL;
  pkv::PrefillLaunch a;
  a.kv_map = &pool->kv_map;
  a.kv16_map = &pool->kv16_map;
  a.pool = static_cast<const uint8_t*>(pool->storage);
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.q_rot = q_rot;
  a.out = out;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.cu_tokens = cu_tokens;
  a.start_pos = start_pos;
  a.batch = batch;
  a.total_tokens = total_tokens;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.rope_table = rope_table;
  a.rope_positions = rope_positions;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.sm_count = sms;
  a.err = pool->d_err;
  e = pkv::launch_prefill(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int paged_gqa_decode_partials(const pkv_pool_t* pool, const float* q_rot,
                              const int32_t* block_tables, int max_blocks,
                              const int32_t* seq_lens, int batch, int num_q_heads, float scale,
                              int pages_per_split, float* o_part, float* lse_part,
                              int32_t* num_splits, int max_splits, void* stream) {
  if (!decode_shape_ok(pool, batch, num_q_heads, max_blocks) || pages_per_split < 1 ||
      !std::isfinite(scale))
    return -EINVAL;
  if (max_splits < max_blocks / pages_per_split + 2) return -EINVAL;
  if (batch == 0) return 0;
  if (!q_rot || !block_tables || !seq_lens || !o_part || !lse_part || !num_splits)
    return -EINVAL;
  if (!aligned16(q_rot) || !aligned16(o_part)) return -EINVAL;
  pkv::DecodeLaunch a = {};
  a.kv_map = &pool->kv_map;
  a.pool = static_cast<const uint8_t*>(pool->storage);
  a.num_pages = pool->num_pages;
  a.num_kv_heads = pool->num_kv_heads;
  a.q_rot = q_rot;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.pages_per_split = pages_per_split;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.num_splits = num_splits;
  a.max_splits = max_splits;
  a.err = pool->d_err;
  a.merge_looks = pool->merge_looks;
  cudaError_t e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int paged_kv_split_combine(const float* o_part, const float* lse_part, const int32_t* num_splits,
                           float* out, int rows, int max_splits, int head_dim, void* stream) {
  if (rows < 0 || max_splits < 1 || head_dim < 1 || head_dim > 1024) return -EINVAL;
  if (rows == 0) return 0;
  if (!o_part || !lse_part || !num_splits || !out) return -EINVAL;
  cudaError_t e = pkv::launch_split_combine(o_part, lse_part, num_splits, out, rows, max_splits,
                                            head_dim, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? 0 : cuda_fail(e);
}

int pkv_get_error(pkv_pool_t* pool, int* bits, int reset) {
  if (!pool || !bits) return -EINVAL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  int v = 0;
  e = cudaMemcpy(&v, pool->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  *bits = v;
  if (reset) {
    e = cudaMemset(pool->d_err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return 0;
}

int pkv_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
