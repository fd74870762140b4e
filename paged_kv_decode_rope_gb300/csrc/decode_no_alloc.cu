// decode_no_alloc.cu -- paged_gqa_decode_no_alloc: the split-KV decode with its
// workspace in a fixed device array instead of caller-provided memory.
//
// Some callers cannot call cudaMalloc: code running under a host framework
// whose memory manager owns all device memory and forbids direct allocation
// (a cudaMalloc there would synchronise the device and bypass the manager's
// accounting), or a plugin that a runtime only hands its input and output
// buffers. For them this entry point takes no workspace argument and never
// allocates: the decode's scratch (the partial results of segments split
// between CTAs, each word tagged so that zero means "not written in this
// call") lives in g_decode_scratch, a file-scope array that every GPU which
// loads this library holds until the process exits.
#include <cerrno>
#include <cmath>
#include <mutex>

#include "../../include/pkv.h"
#include "pkv_internal.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[PKV_NO_ALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};  // device address of g_decode_scratch, per device

// The array's name is a host-side stand-in in host code; a kernel needs its
// device address, looked up once per device with that device current and
// kept for the process (it does not survive a reset of the device's primary
// context).
cudaError_t scratch_address(int device, void** ptr) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[device] = p;
  }
  *ptr = g_scratch_ptr[device];
  return cudaSuccess;
}

}  // namespace

extern "C" int paged_gqa_decode_no_alloc(const pkv_pool_t* pool, const float* q_rot, float* out,
                                         const int32_t* block_tables, int max_blocks,
                                         const int32_t* seq_lens, int batch, int num_q_heads,
                                         float scale, int pages_per_split, void* stream) {
  if (!pool || batch < 0 || max_blocks < 1 || num_q_heads < 1 || pages_per_split < 0 ||
      !std::isfinite(scale) || num_q_heads % pool->num_kv_heads)
    return -EINVAL;
  if (batch == 0) return 0;
  if (!q_rot || !out || !block_tables || !seq_lens) return -EINVAL;
  const size_t need = paged_gqa_decode_workspace_bytes(batch, num_q_heads, pool->num_kv_heads,
                                                       max_blocks, pages_per_split);
  if (need == 0) return -EINVAL;
  if (need > PKV_NO_ALLOC_SCRATCH_BYTES) return -E2BIG;  // sizes beyond the fixed array
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  void* scratch = nullptr;
  if (e == cudaSuccess) e = scratch_address(device, &scratch);
  // The decode reads a zero word as "not written in this call". A call that
  // completes leaves every word it wrote at zero again, but one whose merger
  // gave up waiting (PKV_ERR_TIMEOUT) leaves its partials behind, and this
  // array's callers have no handle to clear it. So every call clears the
  // bytes it will use, on its own stream, before the decode; a memset
  // allocates nothing.
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    pkv::record_cuda_error(e);
    return -EIO;
  }
  return paged_gqa_decode(pool, q_rot, out, block_tables, max_blocks, seq_lens, batch, num_q_heads,
                          scale, pages_per_split, scratch, PKV_NO_ALLOC_SCRATCH_BYTES, stream);
}
