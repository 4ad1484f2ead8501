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
// columns 4 lane + 128 j .. +3 (j = 0, 1) of every split, so a warp access is
// contiguous (512 bytes for fp32 partials, 256 for bf16); the loads of the
// first splits are in flight with the split weights and later ones eight at
// a time, and the gate and the output move as 8-byte bf16x4 accesses.  Two
// partial formats: fp32 (the public entry point) and bf16 (what the
// attention kernel writes for its own splits).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kCombineThreads = 256;

// Partial formats: the raw value a lane loads for four columns, and its
// conversion to fp32 (bf16 -> fp32 is exact).
template <bool kBf16>
struct Partial;
template <>
struct Partial<false> {
  using Elem = float;
  using Raw = float4;
  static constexpr int kMaxFirst = 12;
  __device__ static Raw load(const Elem* p) { return ld_dep_f4_stream(reinterpret_cast<const float4*>(p)); }
  __device__ static Raw zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ static float4 f4(Raw r) { return r; }
};
template <>
struct Partial<true> {
  using Elem = __nv_bfloat16;
  using Raw = uint2;
  static constexpr int kMaxFirst = 16;
  __device__ static Raw load(const Elem* p) { return ld_dep_u2_stream(p); }
  __device__ static Raw zero() { return make_uint2(0u, 0u); }
  __device__ static float4 f4(Raw r) {
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
  }
};

__device__ __forceinline__ void fma4(float4& acc, float w, float4 v) {
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

// Partial addressing.  Uniform splits: split s of row `row` is slot s, row
// `row` of a [S][rows] table.  Balanced plan (plan_splits != NULL): request r
// = row / Mq owns slots plan_base[r] .. + plan_splits[r] - 1 of a [slots][Mq]
// table, and a request with one piece was finished by the attention kernel.
// Wave mode (wave_k >= 0): request r >= wave_k owns slots (r - wave_k) S ..
// + S - 1 of a [slots][Mq] table; the grid covers rows row_begin.. only.
// kFirst: splits whose partials are loaded with the weights (chosen from S at
// launch, so that few splits keep few registers and many warps resident).
template <bool kBf16, int kFirst>
__global__ void __launch_bounds__(kCombineThreads)
    lse_combine_kernel(const typename Partial<kBf16>::Elem* __restrict__ part_o,
                       const float* __restrict__ part_lse,
                       int S_uniform, long long rows, const __nv_bfloat16* __restrict__ gate,
                       __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out,
                       const int* plan_splits, const int* plan_base, int Mq, int gate_dim,
                       long long row_begin, int wave_k) {
  // one warp per half row (256 columns): lane owns columns 128j + 4 lane .. +3, j = 0, 1
  const int lane = threadIdx.x & 31;
  const long long hrow = (long long)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
  if (hrow >= 2 * (rows - row_begin)) return;
  const long long row = row_begin + (hrow >> 1);
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
  } else if (wave_k >= 0) {
    const long long rq = row / Mq;
    slot0 = (rq - wave_k) * S;
    slot_rows = Mq;
    rin = row - rq * Mq;
  }

  // split weights: lane s holds lse_s for s = lane and lane + 32.  The
  // partials of the first kFirst splits are loaded in the same round trip
  // (every split's partial is written, as zeros when its range is empty, so
  // they can be read before the weights are known).
  using P = Partial<kBf16>;
  // debug build (no status word here: a failure is reported by its line)
  SV_DCHECK(S >= 1 && S <= SV_MAX_SPLITS && rin >= 0 && rin < slot_rows && slot0 >= 0 && row < rows &&
                col0 + 128 + 4 <= 512, nullptr);
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < S) l0 = ld_dep_f32(part_lse + (slot0 + lane) * slot_rows + rin);
  if (lane + 32 < S) l1 = ld_dep_f32(part_lse + (slot0 + lane + 32) * slot_rows + rin);
  typename P::Raw v0[kFirst][2];
#pragma unroll
  for (int u = 0; u < kFirst; ++u) {
    const auto* src = part_o + ((slot0 + min(u, S - 1)) * slot_rows + rin) * 512 + col0;
#pragma unroll
    for (int j = 0; j < 2; ++j) v0[u][j] = (u < S) ? P::load(src + 128 * j) : P::zero();
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
      for (int j = 0; j < 2; ++j) fma4(acc[j], ws, P::f4(v0[u][j]));
    }
    // further splits, kRound per round: all their loads in flight before any FMA
    constexpr int kRound = kFirst < 8 ? kFirst : 8;
    for (int s0 = kFirst; s0 < S; s0 += kRound) {
      typename P::Raw v[kRound][2];
      float ws[kRound];
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
        const int s = s0 + u;
        ws[u] = (s < S) ? __shfl_sync(0xFFFFFFFFu, s < 32 ? w0 : w1, s & 31) * inv_z : 0.f;
        const auto* src = part_o + ((slot0 + min(s, S - 1)) * slot_rows + rin) * 512 + col0;
#pragma unroll
        for (int j = 0; j < 2; ++j) v[u][j] = (ws[u] != 0.f) ? P::load(src + 128 * j) : P::zero();
      }
#pragma unroll
      for (int u = 0; u < kRound; ++u) {
#pragma unroll
        for (int j = 0; j < 2; ++j) fma4(acc[j], ws[u], P::f4(v[u][j]));
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

// Internal launcher shared with mla_verify_decode (no argument checks);
// part_o is fp32, or bf16 when bf16_partials.
cudaError_t launch_lse_combine(const void* part_o, bool bf16_partials, const float* part_lse, int S,
                               long long rows, const void* gate, void* out, float* lse,
                               cudaStream_t stream, const int* plan_splits, const int* plan_base,
                               int Mq, int gate_dim, long long row_begin, int wave_k) {
  if (rows - row_begin <= 0) return cudaSuccess;
  const long long blocks = (2 * (rows - row_begin) + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
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
  const auto* g = static_cast<const __nv_bfloat16*>(gate);
  auto* o = static_cast<__nv_bfloat16*>(out);
  // the balanced plan's split counts are only known on the device: the
  // instance that loads four splits with the weights (57 registers, so many
  // warps stay resident) and takes any further ones four at a time; on the
  // long-context c4 batch (2-4 pieces per request) 369.8 -> 361.1 us for the
  // attention call against the 16-split instance (98 registers)
  const int s_max = plan_splits ? 4 : S;
  auto launch = [&](auto kernel, const auto* po) {
    return cudaLaunchKernelEx(&cfg, kernel, po, part_lse, S, rows, g, o, lse, plan_splits, plan_base,
                              Mq, gate_dim, row_begin, wave_k);
  };
  cudaError_t e;
  if (bf16_partials) {
    const auto* po = static_cast<const __nv_bfloat16*>(part_o);
    e = s_max <= 4 ? launch(lse_combine_kernel<true, 4>, po)
        : s_max <= 8 ? launch(lse_combine_kernel<true, 8>, po)
                     : launch(lse_combine_kernel<true, Partial<true>::kMaxFirst>, po);
  } else {
    const auto* po = static_cast<const float*>(part_o);
    e = s_max <= 4 ? launch(lse_combine_kernel<false, 4>, po)
        : s_max <= 8 ? launch(lse_combine_kernel<false, 8>, po)
                     : launch(lse_combine_kernel<false, Partial<false>::kMaxFirst>, po);
  }
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
  return sv::launch_lse_combine(part_o, false, part_lse, S, rows, gate, out, lse,
                                reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr,
                                1, SV_LATENT_DIM, 0, -1) == cudaSuccess
             ? SV_OK
             : SV_ERR_LAUNCH;
}
