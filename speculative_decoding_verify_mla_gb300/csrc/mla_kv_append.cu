// mla_kv_append.cu - write the latent rows of the verify tokens into the paged
// KV cache before the attention reads them.
//
// Definition (the per-token KV write slot of "TensorRT-LLM PR #18166: Kimi K3
// DSpark speculative decoding under Helix CP", first commit message: global
// position -> rank-local write slot, -1 = not owned; on one GPU every position
// is owned): token t of request r = t / q_per_req with position pos >= 0
// stores its 512-wide latent row in page block_table[r][pos / 64], slot
// pos % 64; pos = -1 skips the token.
//
// HBM-bound byte copy: one warp per token row (1 KB), each lane moves two
// 16-byte words, so a warp writes one whole latent row.
#include <cuda_runtime.h>

#include <cstdint>

#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(const uint4* __restrict__ kv_new, const int32_t* __restrict__ positions,
                     const int32_t* __restrict__ block_table, int T, int q_per_req, int max_pages,
                     uint4* __restrict__ kv_pages, int num_pages, int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int pos = __ldg(positions + t);
  if (pos < 0) return;
  if (pos >= max_pages * SV_PAGE_SIZE) {
    if (lane == 0 && status) atomicOr(status, SV_DEV_BAD_BOUND);
    return;
  }
  const int r = t / q_per_req;
  const int page = __ldg(block_table + (long long)r * max_pages + pos / SV_PAGE_SIZE);
  if (page < 0 || page >= num_pages) {
    if (lane == 0 && status) atomicOr(status, SV_DEV_BAD_PAGE);
    return;
  }
  // a latent row is 512 bf16 = 64 x 16 bytes
  const uint4* src = kv_new + (long long)t * 64;
  uint4* dst = kv_pages + ((long long)page * SV_PAGE_SIZE + pos % SV_PAGE_SIZE) * 64;
  const uint4 a = __ldg(src + lane);
  const uint4 b = __ldg(src + 32 + lane);
  dst[lane] = a;
  dst[32 + lane] = b;
}

}  // namespace
}  // namespace sv

extern "C" sv_status mla_kv_append(const void* kv_new, const int32_t* positions,
                                   const int32_t* block_table, int R, int q_per_req,
                                   int max_pages_per_req, void* kv_pages, int num_pages,
                                   int page_size, int32_t* status, sv_stream_t stream) {
  if (R < 0 || q_per_req < 1 || max_pages_per_req < 0 || num_pages < 0) return SV_ERR_SHAPE;
  if (page_size != SV_PAGE_SIZE) return SV_ERR_UNSUPPORTED;
  const long long T = (long long)R * q_per_req;
  if (T == 0) return SV_OK;
  if (T > 0x7FFFFFFFll - 8 || max_pages_per_req < 1 || num_pages < 1) return SV_ERR_SHAPE;
  if (!kv_new || !positions || !block_table || !kv_pages) return SV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(kv_new) & 15u) || (reinterpret_cast<uintptr_t>(kv_pages) & 15u) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return SV_ERR_ALIGN;
  const long long blocks = (T + (sv::kAppendThreads / 32) - 1) / (sv::kAppendThreads / 32);
  sv::kv_append_kernel<<<(unsigned)blocks, sv::kAppendThreads, 0,
                         reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(kv_new), positions, block_table, (int)T, q_per_req,
      max_pages_per_req, static_cast<uint4*>(kv_pages), num_pages, status);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_LAUNCH;
}
