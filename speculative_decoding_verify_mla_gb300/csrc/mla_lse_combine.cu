// mla_lse_combine.cu - LSE merge of split-KV attention partials + sigmoid gate.
//
// Definition (the CP / DCP merge of "TensorRT-LLM PR #18166: Kimi K3 DSpark
// speculative decoding under Helix CP", second and third commit messages, and
// of the vLLM page "kimi_k3/nvidia/specialized_decode/drafter/model"):
//   lse = ln sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) * o_s,
//   out = sigmoid(gate) * o  (bf16, round to nearest even).
// A row whose partials are all -inf gets lse = -inf and out = 0: the weight of
// an empty partial is exactly 0 and its o_s is never read, so a zero-bound
// row cannot poison the merge with 0 * NaN.
//
// HBM-bound: one warp per (token, head) row; each lane owns 16 of the 512
// columns as four float4 (coalesced 512-byte warp accesses per split), the
// gate and the output move as 8-byte bf16x4 accesses.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"

namespace sv {
namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + __expf(-g)); }

__global__ void __launch_bounds__(kCombineThreads)
    lse_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                       int S, long long rows, const __nv_bfloat16* __restrict__ gate,
                       __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;

  // split weights: lane s holds lse_s for s = lane and lane + 32
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < S) l0 = __ldg(part_lse + (long long)lane * rows + row);
  if (lane + 32 < S) l1 = __ldg(part_lse + (long long)(lane + 32) * rows + row);
  float m = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));

  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse_row = -INFINITY;
  if (m != -INFINITY) {
    const float w0 = (l0 == -INFINITY) ? 0.f : __expf(l0 - m);
    const float w1 = (l1 == -INFINITY) ? 0.f : __expf(l1 - m);
    float z = w0 + w1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    const float inv_z = 1.0f / z;
    lse_row = m + __logf(z);
    for (int s = 0; s < S; ++s) {
      const float ws = __shfl_sync(0xFFFFFFFFu, s < 32 ? w0 : w1, s & 31) * inv_z;
      if (ws == 0.f) continue;  // warp-uniform: an empty or negligible split is never read
      const float4* src = reinterpret_cast<const float4*>(part_o + ((long long)s * rows + row) * 512);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 v = __ldcs(src + lane + 32 * j);
        acc[j].x = fmaf(ws, v.x, acc[j].x);
        acc[j].y = fmaf(ws, v.y, acc[j].y);
        acc[j].z = fmaf(ws, v.z, acc[j].z);
        acc[j].w = fmaf(ws, v.w, acc[j].w);
      }
    }
  }
  const uint2* g2 = reinterpret_cast<const uint2*>(gate + row * 512);
  uint2* o2 = reinterpret_cast<uint2*>(out + row * 512);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint2 graw = __ldg(g2 + lane + 32 * j);
    const float2 ga = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.x));
    const float2 gb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.y));
    const __nv_bfloat162 r0 = __floats2bfloat162_rn(sigmoidf_(ga.x) * acc[j].x, sigmoidf_(ga.y) * acc[j].y);
    const __nv_bfloat162 r1 = __floats2bfloat162_rn(sigmoidf_(gb.x) * acc[j].z, sigmoidf_(gb.y) * acc[j].w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&r0);
    packed.y = *reinterpret_cast<const uint32_t*>(&r1);
    o2[lane + 32 * j] = packed;
  }
  if (lane == 0) lse_out[row] = lse_row;
}

}  // namespace

// Internal launcher shared with mla_verify_decode (no argument checks).
cudaError_t launch_lse_combine(const float* part_o, const float* part_lse, int S, long long rows,
                               const void* gate, void* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
  lse_combine_kernel<<<(unsigned)blocks, kCombineThreads, 0, stream>>>(
      part_o, part_lse, S, rows, static_cast<const __nv_bfloat16*>(gate),
      static_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}

}  // namespace sv

extern "C" sv_status mla_lse_combine(const float* part_o, const float* part_lse, int S, int T,
                                     int H, const void* gate, void* out, float* lse,
                                     sv_stream_t stream) {
  if (T < 0 || H < 0) return SV_ERR_SHAPE;
  if (S < 1 || S > SV_MAX_SPLITS) return SV_ERR_SHAPE;
  const long long rows = (long long)T * H;
  if (rows == 0) return SV_OK;
  if (rows > (1ll << 31) * (256 / 32)) return SV_ERR_SHAPE;
  if (!part_o || !part_lse || !gate || !out || !lse) return SV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(part_o) & 15u) || (reinterpret_cast<uintptr_t>(part_lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(gate) & 7u) || (reinterpret_cast<uintptr_t>(out) & 7u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return SV_ERR_ALIGN;
  return sv::launch_lse_combine(part_o, part_lse, S, rows, gate, out, lse,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SV_OK
             : SV_ERR_LAUNCH;
}
