// mla_wuv_project.cu - per-head value up-projection of the absorbed MLA
// output: v[t][h][:] = W_UV[h] @ x[t][h][:], x the gated 512-wide latent
// output of the attention (after the LSE merge), W_UV[h] of shape
// [v_dim][512] ("LSE combine + W_UV" after the context-parallel merge on the
// vLLM page "kimi_k3/nvidia/specialized_decode/drafter/model"; absorbed MLA
// keeps W_UV out of the attention itself).
//
// One CTA per (head, 128-token tile): a tcgen05 GEMM with M = 128 tokens,
// N = v_dim, K = 512.  A (the tokens' latent rows of head h, stride H*512)
// and B (W_UV[h]) arrive by TMA in eight 64-column K chunks through a ring
// of as many stages as shared memory holds for this v_dim (7 at v_dim 128,
// so nearly all chunks are in flight at once; 128-byte swizzle, K-major);
// the accumulator lives in TMEM
// and the epilogue converts it to bf16 and stores one token row per thread.
// Warp 0: TMEM allocation and the TMA producer (lane 0); warp 1 lane 0: MMA
// issue; all four warps: epilogue.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sv_host.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kWThreads = 128;
constexpr int kWMaxStages = 8;
constexpr int kWChunks = SV_LATENT_DIM / 64;  // K chunks of 64 columns
constexpr int kWMaxV = 256;                    // N of one MMA
constexpr int kWABytes = 128 * 128;            // 128 token rows x 64 bf16
constexpr int kWSmemMax = 227 * 1024;          // dynamic shared memory of one CTA
constexpr int kWTail = 8 * (2 * kWMaxStages + 1) + 16;  // barriers, TMEM slot, abort flag

// Stage bytes (A chunk + B chunk, 1024-aligned) and the number of stages that
// fit for a given v_dim; both the launch and the kernel use them.
__host__ __device__ constexpr int wuv_stage_bytes(int v_dim) {
  return (kWABytes + v_dim * 128 + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int wuv_stages(int v_dim) {
  return (kWSmemMax - 1024 - kWTail) / wuv_stage_bytes(v_dim) < kWMaxStages
             ? (kWSmemMax - 1024 - kWTail) / wuv_stage_bytes(v_dim)
             : kWMaxStages;
}
__host__ __device__ constexpr int wuv_smem_bytes(int v_dim) {
  return wuv_stages(v_dim) * wuv_stage_bytes(v_dim) + kWTail + 1024;
}

// kShortWaits: the test instance, whose bounded waits give up after wait_ns
// instead of kWaitTimeoutNs.
template <bool kShortWaits>
__global__ void __launch_bounds__(kWThreads, 1)
    wuv_project_kernel(const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w, int T, int H, int v_dim,
                       __nv_bfloat16* __restrict__ out_v, int32_t* __restrict__ status, uint64_t wait_ns) {
  const uint64_t limit = kShortWaits ? wait_ns : kWaitTimeoutNs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* const sptr = smem_raw + (sbase - raw);
  const int kWStages = wuv_stages(v_dim);
  const int kWStageBytes = wuv_stage_bytes(v_dim);
  const uint32_t bar0 = sbase + kWStages * kWStageBytes;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kWMaxStages + s); };
  const uint32_t done = bar0 + 8u * (2 * kWMaxStages);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sptr + kWStages * kWStageBytes + 8 * (2 * kWMaxStages + 1));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * 128;
  const uint32_t tmem_cols = v_dim <= 32 ? 32u : (v_dim <= 64 ? 64u : (v_dim <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t b_bytes = (uint32_t)v_dim * 128u;

  if (warp == 0) {
    // ---- TMA producer: chunk c of A (tokens t0.., columns 64c..) and of B
    if (lane == 0) {
      int last[kWMaxStages] = {-1, -1, -1, -1, -1, -1, -1, -1};
      for (int c = 0; c < kWChunks; ++c) {
        const int s = c % kWStages, rd = c / kWStages;
        if (rd > 0 && !mbar_wait<false>(empty(s), (rd - 1) & 1, abort_flag, status, limit)) break;
        mbar_arrive_expect_tx(full(s), kWABytes + b_bytes);
        const uint32_t st = sbase + s * kWStageBytes;
        tma_load_3d(st, &tmap_x, full(s), c * 64, h, t0);
        tma_load_3d(st + kWABytes, &tmap_w, full(s), c * 64, 0, h);
        last[s] = rd;
      }
      // every copy has landed before teardown
      for (int s = 0; s < kWStages; ++s) {
        if (last[s] < 0) continue;
        const uint64_t tw = globaltimer_ns();
        while (!mbar_test(full(s), last[s] & 1) && globaltimer_ns() - tw < kWaitTimeoutNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issue: D[128 x v] += A[128 x 16] B[v x 16]^T, 4 per chunk
    const uint32_t idesc = idesc_bf16_f32(128, v_dim, false, false);
    bool ok = true;
    for (int c = 0; ok && c < kWChunks; ++c) {
      const int s = c % kWStages, rd = c / kWStages;
      ok = mbar_wait<false>(full(s), rd & 1, abort_flag, status, limit);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = sbase + s * kWStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc_sw128(st + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(st + kWABytes + kk * 32, 16, 1024);
          mma_ss(tmem, ad, bd, idesc, (c > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(empty(s));
      }
      __syncwarp();
    }
    if (lane == 0) {
      mma_commit(done);
      // the MMAs issued have completed before the CTA moves on to the
      // epilogue and frees the TMEM, also when a wait gave up
      const uint64_t tw = globaltimer_ns();
      while (!mbar_test(done, 0) && globaltimer_ns() - tw < kWaitTimeoutNs) {
      }
    }
    __syncwarp();
  }

  // ---- epilogue: thread i owns token row t0 + i (TMEM lane i).  After the
  // barrier every role has finished: a CTA in which a wait gave up (its
  // abort flag is set, and the MMAs may not have run) reads no TMEM and
  // writes nothing.
  __syncthreads();
  const bool ok =
      __all_sync(0xFFFFFFFFu, mbar_wait<false>(done, 0, abort_flag, status, limit) && *abort_flag == 0);
  tc_fence_after();
  const int t = t0 + warp * 32 + lane;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  for (int c0 = 0; ok && c0 < v_dim; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(tmem + lane_off + (uint32_t)c0, v);
    tmem_wait_ld();
    if (t < T) {
      uint4* dst = reinterpret_cast<uint4*>(out_v + ((long long)t * H + h) * v_dim + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
        w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
        w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
        w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
        dst[q] = w;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

std::mutex g_wuv_mu;
bool g_wuv_attr[64];

sv_status wuv_impl(const void* x, const void* w_uv, int T, int H, int v_dim, void* out_v, int32_t* status,
                   sv_stream_t stream, uint64_t wait_ns) {
  if (T < 0 || H < 0) return SV_ERR_SHAPE;
  if (v_dim < 32 || v_dim > kWMaxV || v_dim % 32 != 0) return SV_ERR_UNSUPPORTED;
  if (T == 0 || H == 0) return SV_OK;
  if ((long long)T * H > 0x7FFFFFFFll) return SV_ERR_SHAPE;
  if (!x || !w_uv || !out_v) return SV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_uv) & 15u) ||
      (reinterpret_cast<uintptr_t>(out_v) & 15u))
    return SV_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_DEVICE;
  {
    std::lock_guard<std::mutex> lk(g_wuv_mu);
    if (!g_wuv_attr[dev]) {
      if (cudaFuncSetAttribute(wuv_project_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kWSmemMax) != cudaSuccess ||
          cudaFuncSetAttribute(wuv_project_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kWSmemMax) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_DEVICE;
      }
      g_wuv_attr[dev] = true;
    }
  }
  CUtensorMap tmap_x, tmap_w;
  const cuuint64_t x_dims[3] = {(cuuint64_t)SV_LATENT_DIM, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint32_t x_box[3] = {64, 1, 128};
  const cuuint64_t w_dims[3] = {(cuuint64_t)SV_LATENT_DIM, (cuuint64_t)v_dim, (cuuint64_t)H};
  const cuuint32_t w_box[3] = {64, (cuuint32_t)v_dim, 1};
  const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_map(&tmap_x, bf16, 2, x, 3, x_dims, x_box) ||
      !encode_map(&tmap_w, bf16, 2, w_uv, 3, w_dims, w_box))
    return get_encode_fn() ? SV_ERR_ALIGN : SV_ERR_DEVICE;
  const dim3 grid((unsigned)H, (unsigned)((T + 127) / 128), 1);
  auto kernel = wait_ns < kWaitTimeoutNs ? wuv_project_kernel<true> : wuv_project_kernel<false>;
  kernel<<<grid, kWThreads, wuv_smem_bytes(v_dim), reinterpret_cast<cudaStream_t>(stream)>>>(
      tmap_x, tmap_w, T, H, v_dim, static_cast<__nv_bfloat16*>(out_v), status, wait_ns);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_LAUNCH;
}

}  // namespace
}  // namespace sv

extern "C" sv_status mla_wuv_project(const void* x, const void* w_uv, int T, int H, int v_dim,
                                     void* out_v, int32_t* status, sv_stream_t stream) {
  return sv::wuv_impl(x, w_uv, T, H, v_dim, out_v, status, stream, sv::kWaitTimeoutNs);
}

// Test entry point: mla_wuv_project with the limit of every bounded wait of
// the kernel lowered to wait_ns (the drains before teardown keep theirs).
extern "C" sv_status sv_test_mla_wuv_project_wait_limit(const void* x, const void* w_uv, int T, int H, int v_dim,
                                                        void* out_v, int32_t* status, sv_stream_t stream,
                                                        uint64_t wait_ns) {
  if (wait_ns > sv::kWaitTimeoutNs) return SV_ERR_SHAPE;  // it only shortens the waits
  return sv::wuv_impl(x, w_uv, T, H, v_dim, out_v, status, stream, wait_ns);
}
