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
// HBM-bound: one warp per half row (256 of the 512 columns); each lane owns
// two float4 of every split (coalesced 512-byte warp accesses), the loads of
// eight splits are in flight before their FMAs, and the gate and the output
// move as 8-byte bf16x4 accesses.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kCombineThreads = 256;

// Partial addressing.  Uniform splits: split s of row `row` is slot s, row
// `row` of a [S][rows] table.  Balanced plan (plan_splits != NULL): request r
// = row / Mq owns slots plan_base[r] .. + plan_splits[r] - 1 of a [slots][Mq]
// table, and a request with one piece was finished by the attention kernel.
__global__ void __launch_bounds__(kCombineThreads)
    lse_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                       int S_uniform, long long rows, const __nv_bfloat16* __restrict__ gate,
                       __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out,
                       const int* plan_splits, const int* plan_base, int Mq, int gate_dim) {
  // one warp per half row (256 columns): lane owns columns 128j + 4 lane .. +3, j = 0, 1
  const int lane = threadIdx.x & 31;
  const long long hrow = (long long)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
  if (hrow >= 2 * rows) return;
  const long long row = hrow >> 1;
  const int col0 = (int)(hrow & 1) * 256 + 4 * lane;
  // the gate does not depend on the attention kernel: fetch it first
  // (elementwise [T][H][512], or one value per row when head-wise)
  uint2 graw[2] = {make_uint2(0u, 0u), make_uint2(0u, 0u)};
  float g_row = 0.f;
  if (gate_dim == 1) {
    g_row = fast_sigmoid(__bfloat162float(gate[row]));
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      graw[j] = __ldg(reinterpret_cast<const uint2*>(gate + row * 512 + col0 + 128 * j));
  }
  // when launched behind the attention kernel (programmatic dependent
  // launch), wait here until its partials are complete and visible
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int S = S_uniform;
  long long slot0 = 0, slot_rows = rows, rin = row;
  if (plan_splits) {
    const long long rq = row / Mq;
    S = ld_dep_s32(plan_splits + rq);
    if (S < 2) return;  // finished by the attention kernel
    slot0 = ld_dep_s32(plan_base + rq);
    slot_rows = Mq;
    rin = row - rq * Mq;
  }

  // split weights: lane s holds lse_s for s = lane and lane + 32.  The
  // partials of the first kFirst splits are loaded in the same round trip
  // (every split's partial is written, as zeros when its range is empty, so
  // they can be read before the weights are known).
  constexpr int kFirst = 12;
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < S) l0 = ld_dep_f32(part_lse + (slot0 + lane) * slot_rows + rin);
  if (lane + 32 < S) l1 = ld_dep_f32(part_lse + (slot0 + lane + 32) * slot_rows + rin);
  float4 v0[kFirst][2];
#pragma unroll
  for (int u = 0; u < kFirst; ++u) {
    const float* src = part_o + ((slot0 + min(u, S - 1)) * slot_rows + rin) * 512 + col0;
#pragma unroll
    for (int j = 0; j < 2; ++j)
      v0[u][j] = (u < S) ? ld_dep_f4_stream(reinterpret_cast<const float4*>(src + 128 * j))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));

  float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  float lse_row = -INFINITY;
  if (m != -INFINITY) {
    const float w0 = (l0 == -INFINITY) ? 0.f : __expf(l0 - m);
    const float w1 = (l1 == -INFINITY) ? 0.f : __expf(l1 - m);
    float z = w0 + w1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    const float inv_z = 1.0f / z;
    lse_row = m + __logf(z);
#pragma unroll
    for (int u = 0; u < kFirst; ++u) {
      const float ws = (u < S) ? __shfl_sync(0xFFFFFFFFu, w0, u) * inv_z : 0.f;
      if (ws == 0.f) continue;  // an empty split's values are never used (0 * NaN stays out)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        acc[j].x = fmaf(ws, v0[u][j].x, acc[j].x);
        acc[j].y = fmaf(ws, v0[u][j].y, acc[j].y);
        acc[j].z = fmaf(ws, v0[u][j].z, acc[j].z);
        acc[j].w = fmaf(ws, v0[u][j].w, acc[j].w);
      }
    }
    // further splits, eight per round: all their loads in flight before any FMA
    for (int s0 = kFirst; s0 < S; s0 += 8) {
      float4 v[8][2];
      float ws[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + u;
        ws[u] = (s < S) ? __shfl_sync(0xFFFFFFFFu, s < 32 ? w0 : w1, s & 31) * inv_z : 0.f;
        const float* src = part_o + ((slot0 + min(s, S - 1)) * slot_rows + rin) * 512 + col0;
#pragma unroll
        for (int j = 0; j < 2; ++j)
          v[u][j] = (ws[u] != 0.f) ? ld_dep_f4_stream(reinterpret_cast<const float4*>(src + 128 * j))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acc[j].x = fmaf(ws[u], v[u][j].x, acc[j].x);
          acc[j].y = fmaf(ws[u], v[u][j].y, acc[j].y);
          acc[j].z = fmaf(ws[u], v[u][j].z, acc[j].z);
          acc[j].w = fmaf(ws[u], v[u][j].w, acc[j].w);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 ga = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw[j].x));
    const float2 gb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw[j].y));
    const bool hw = (gate_dim == 1);
    const __nv_bfloat162 r0 = __floats2bfloat162_rn((hw ? g_row : fast_sigmoid(ga.x)) * acc[j].x,
                                                    (hw ? g_row : fast_sigmoid(ga.y)) * acc[j].y);
    const __nv_bfloat162 r1 = __floats2bfloat162_rn((hw ? g_row : fast_sigmoid(gb.x)) * acc[j].z,
                                                    (hw ? g_row : fast_sigmoid(gb.y)) * acc[j].w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&r0);
    packed.y = *reinterpret_cast<const uint32_t*>(&r1);
    *reinterpret_cast<uint2*>(out + row * 512 + col0 + 128 * j) = packed;
  }
  if (lane == 0 && (hrow & 1) == 0) lse_out[row] = lse_row;
}

}  // namespace

// Internal launcher shared with mla_verify_decode (no argument checks).
cudaError_t launch_lse_combine(const float* part_o, const float* part_lse, int S, long long rows,
                               const void* gate, void* out, float* lse, cudaStream_t stream,
                               const int* plan_splits, const int* plan_base, int Mq, int gate_dim) {
  if (rows == 0) return cudaSuccess;
  const long long blocks = (2 * rows + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
  // programmatic dependent launch: the grid may start while the previous
  // kernel on the stream finishes; griddepcontrol.wait guards the partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, lse_combine_kernel, part_o, part_lse, S, rows,
                                           static_cast<const __nv_bfloat16*>(gate),
                                           static_cast<__nv_bfloat16*>(out), lse, plan_splits,
                                           plan_base, Mq, gate_dim);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
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
                                reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr,
                                1, SV_LATENT_DIM) == cudaSuccess
             ? SV_OK
             : SV_ERR_LAUNCH;
}
