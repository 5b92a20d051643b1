// pkv_paged_attention_noalloc: paged attention for callers that must not allocate device
// memory.  The scratch space that pkv_paged_attention takes from a caller-provided
// workspace comes here from a fixed array that lives inside this library.
//
// Who needs this: code that is handed device pointers by a host framework that owns all
// device memory (its own caching allocator or a fixed memory plan) and may not call
// cudaMalloc itself, and latency-critical serving loops that avoid cudaMalloc / cudaFree
// because those calls can block or synchronise the device, or fail in the middle of a step
// when memory is tight.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

// The built-in scratch.  Every GPU that loads this library holds PKV_NOALLOC_SCRATCH_BYTES of
// it until the process exits, and all calls on that GPU share it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_scratch[kMaxDevices];
cudaError_t g_setup_status[kMaxDevices];

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_paged_attention_noalloc(const void* q, int64_t q_st, int64_t q_sh, const void* k_cache,
                                           const void* v_cache, int64_t num_blocks, int64_t block_size,
                                           const int32_t* block_tables, int64_t bt_stride,
                                           int64_t max_blocks_per_seq, const int32_t* context_lens,
                                           const int32_t* query_start_loc, int64_t num_seqs, void* out,
                                           int64_t o_st, int64_t o_sh, int64_t num_tokens, int64_t num_q_heads,
                                           int64_t num_kv_heads, int64_t head_dim, float scale, void* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  // First call on this device (with it current): look up the device address of the array.
  // In host code the array's name only stands in for the symbol; it is not a device address.
  std::call_once(g_once[dev], [dev]() {
    void* p = nullptr;
    g_setup_status[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    g_scratch[dev] = g_setup_status[dev] == cudaSuccess ? p : nullptr;
  });
  if (g_setup_status[dev] != cudaSuccess || g_scratch[dev] == nullptr) return PKV_ERR_CUDA;

  // Sizes whose scratch does not fit the array are refused before anything is launched.
  // (Invalid sizes report 0 here and are rejected by the validation below.)
  const size_t need = pkv_paged_attention_workspace_size(num_tokens, num_seqs, num_q_heads, num_kv_heads,
                                                         head_dim, max_blocks_per_seq);
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;

  // Nothing in the scratch needs clearing: the planner kernel writes every field that the
  // later kernels of the same call read, so a previous call's leftovers are never used.
  return pkv_paged_attention(q, q_st, q_sh, k_cache, v_cache, num_blocks, block_size, block_tables, bt_stride,
                             max_blocks_per_seq, context_lens, query_start_loc, num_seqs, out, o_st, o_sh,
                             num_tokens, num_q_heads, num_kv_heads, head_dim, scale, g_scratch[dev],
                             PKV_NOALLOC_SCRATCH_BYTES, stream);
}
