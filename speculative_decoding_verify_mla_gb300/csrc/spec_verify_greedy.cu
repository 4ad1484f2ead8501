// spec_verify_greedy.cu - greedy verification of drafted tokens with KV trim.
//
// Definition ("M* PR #257: Kimi K3 support with DSpark speculative decoding",
// section "Speculative decoding": verification is greedy, the KV trims the
// rejected tails): a[t] = argmax_v logits[t][v] with the lowest v on ties;
// request r accepts the longest prefix of its k drafts with d_j == a_{j-1};
// next token a_n; kv_lens_out = kv_lens_in - (k - n).
//
// One launch.  The [T][V] fp32 logits are cut into chunks of C floats (about
// twelve CTAs per SM); each CTA streams one chunk with coalesced 128-bit loads
// (about eight in flight per thread: the load of the next round's slot is
// issued as soon as a value is taken), reduces it to a 64-bit key
// (order-preserving value bits << 32 | ~index, so the max key is the max
// value at the lowest index) and folds it into its row's key with a 64-bit
// atomicMax.  (Short CTAs matter when the verify step runs this kernel beside
// the attention: a CTA that finishes soon hands its SM space back to the
// attention's next units.  Twelve per SM against four: the C = 32 verify
// step 79.5 -> 73.3 us on GB300, the calls alone unchanged within 1 us.)
// The CTA that takes the last ticket gives each thread whole requests: it
// reads the request's row keys and drafts in one round trip, decodes the
// argmax ids and writes accepted / next token / trimmed kv_lens, and leaves
// the ticket and every row key zero again.  Nothing waits on another CTA.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "specverify.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kGreedyThreads = 256;
constexpr size_t kGreedyHeader = 256;  // ticket counter, padded

__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 compare equal
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

// Streaming 16-byte load: bypass L1, ask L2 to fetch 256-byte sectors.
__device__ __forceinline__ float4 ld_stream_f4(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, k, o);
    k = other > k ? other : k;
  }
  return k;
}

__global__ void __launch_bounds__(kGreedyThreads)
    greedy_verify_kernel(const float* __restrict__ logits, int T, int V, int R, int k,
                         int chunk, int nchunks, bool vec4,
                         const int32_t* __restrict__ draft_tokens,
                         const int32_t* __restrict__ kv_lens_in, int32_t* __restrict__ argmax_ids,
                         int32_t* __restrict__ accepted, int32_t* __restrict__ next_tokens,
                         int32_t* __restrict__ kv_lens_out, unsigned int* __restrict__ ticket,
                         unsigned long long* row_key) {
  // Shared memory stays under 1 KB so that this kernel can share an SM with
  // the attention kernel (which leaves ~1.8 KB of the SM's shared memory).
  __shared__ unsigned long long s_warp[kGreedyThreads / 32];
  __shared__ bool s_last;
  const int tid = threadIdx.x;
  const long long bid = blockIdx.x;
  const int t = (int)(bid / nchunks);
  const int c = (int)(bid % nchunks);
  const long long lo = (long long)c * chunk;
  const long long hi = min((long long)V, lo + chunk);
  const float* row = logits + (long long)t * V;
  // debug build (no status word here: a failure is reported by its line)
  SV_DCHECK(t >= 0 && t < T && lo >= 0 && lo <= hi && hi <= V, nullptr);

  // ---- chunk scan: each thread walks its elements in increasing index order
  float best_v = -INFINITY;
  uint32_t best_i = 0xFFFFFFFFu;
  if (vec4) {
    const float4* p4 = reinterpret_cast<const float4*>(row + lo);
    const int n4 = (int)((hi - lo) >> 2);
    int i = tid;
    // rounds of eight 16-byte loads per thread, pipelined: as soon as a
    // value is taken, the load of the same slot of the next round is
    // issued, so about eight loads stay in flight per thread without a
    // second buffer (elements are still reduced in increasing index order,
    // which keeps the lowest index on ties)
    constexpr int kRound = 8 * kGreedyThreads;
    if (i + 7 * kGreedyThreads < n4) {
      float4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = ld_stream_f4(p4 + i + u * kGreedyThreads);
      while (true) {
        const int j = i + kRound;
        const bool more = j + 7 * kGreedyThreads < n4;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 v = a[u];
          if (more) a[u] = ld_stream_f4(p4 + j + u * kGreedyThreads);
          const uint32_t base = (uint32_t)(lo + 4ll * (i + u * kGreedyThreads));
          if (best_i == 0xFFFFFFFFu) { best_v = v.x; best_i = base; }
          else if (v.x > best_v) { best_v = v.x; best_i = base; }
          if (v.y > best_v) { best_v = v.y; best_i = base + 1; }
          if (v.z > best_v) { best_v = v.z; best_i = base + 2; }
          if (v.w > best_v) { best_v = v.w; best_i = base + 3; }
        }
        i = j;
        if (!more) break;
      }
    }
    for (; i < n4; i += kGreedyThreads) {
      const float4 a = ld_stream_f4(p4 + i);
      const uint32_t base = (uint32_t)(lo + 4ll * i);
      if (best_i == 0xFFFFFFFFu) { best_v = a.x; best_i = base; }
      else if (a.x > best_v) { best_v = a.x; best_i = base; }
      if (a.y > best_v) { best_v = a.y; best_i = base + 1; }
      if (a.z > best_v) { best_v = a.z; best_i = base + 2; }
      if (a.w > best_v) { best_v = a.w; best_i = base + 3; }
    }
  } else {
    for (long long i = lo + tid; i < hi; i += kGreedyThreads) {
      const float x = __ldcs(row + i);
      if (best_i == 0xFFFFFFFFu || x > best_v) { best_v = x; best_i = (uint32_t)i; }
    }
  }
  unsigned long long key = (best_i == 0xFFFFFFFFu) ? 0ull : argmax_key(best_v, best_i);
  key = warp_max_u64(key);
  if ((tid & 31) == 0) s_warp[tid >> 5] = key;
  __syncthreads();
  if (tid < 32) {
    unsigned long long kk = tid < kGreedyThreads / 32 ? s_warp[tid] : 0ull;
    kk = warp_max_u64(kk);
    if (tid == 0) {
      atomicMax(row_key + t, kk);
      __threadfence();
      s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
    }
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA: one thread per request reads its tokens' row keys and its
  // drafts in one round trip (all loads issued before any is used, eight
  // tokens at a time), decodes the argmax ids, and finds the first token j
  // whose draft differs from a_j (or j = k): accepted = j, next token = a_j,
  // kv_lens_out = kv_lens_in - (k - j).  Every row key and the ticket are
  // left zero for the next call.  The keys were raised with atomics by the
  // other CTAs before their ticket; the reads go to L2 (.cg).
  __threadfence();
  for (int r = tid; r < R; r += kGreedyThreads) {
    const int t0 = r * (k + 1);
    int n = -1, nxt = 0;
    for (int j0 = 0; j0 <= k; j0 += 8) {
      unsigned long long key[8];
      int d[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        SV_DCHECK(j > k || (long long)t0 + j < (long long)T, nullptr);
        key[u] = (j <= k) ? __ldcg(row_key + t0 + j) : 0ull;
        d[u] = (j < k) ? __ldg(draft_tokens + (long long)r * k + j) : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        if (j <= k) {
          const int a = (int)(0xFFFFFFFFu - (uint32_t)(key[u] & 0xFFFFFFFFull));
          argmax_ids[t0 + j] = a;
          row_key[t0 + j] = 0ull;
          if (n < 0 && (j == k || d[u] != a)) {
            n = j;
            nxt = a;
          }
        }
      }
    }
    accepted[r] = n;
    next_tokens[r] = nxt;
    kv_lens_out[r] = kv_lens_in[r] - (k - n);
  }
  if (tid == 0) *ticket = 0u;  // leave the workspace zeroed for the next call
}

// Chunk length (floats) as a function of the problem only.
int greedy_chunk(int T, int V) {
  const long long total = (long long)T * V;
  long long c = (total + 12 * 152 - 1) / (12 * 152);  // about twelve CTAs per SM
  c = (c + 8191) / 8192 * 8192;
  // CTAs of at least 64 KB when the logits can fill four of them per SM:
  // 32 KB CTAs take one round of loads per thread and pay the per-CTA key
  // atomic and ticket for little streaming (the C = 64 decode call 16.2 ->
  // 14.5 us; smaller batches keep 32 KB chunks to spread over the SMs)
  const long long cmin = total >= 4ll * 152 * 16384 ? 16384 : 8192;
  if (c < cmin) c = cmin;
  if (c > 65536) c = 65536;
  return (int)c;
}

}  // namespace
}  // namespace sv

// Workspace: ticket header, then the row keys [T]; all zero at rest.
extern "C" size_t sv_greedy_workspace_bytes(int T, int V) {
  if (T <= 0 || V <= 0) return sv::kGreedyHeader;
  return sv::kGreedyHeader + (size_t)T * sizeof(unsigned long long);
}

namespace sv {
namespace {

// Host-side checks of everything but the workspace, shared by both greedy
// entry points so that a failed check enqueues nothing in either.  SV_OK with
// *empty = true: T == 0, nothing to do.
sv_status greedy_check(const float* logits, int T, int V, int R, int k, const int32_t* draft_tokens,
                       const int32_t* kv_lens_in, const int32_t* argmax_ids, const int32_t* accepted,
                       const int32_t* next_tokens, const int32_t* kv_lens_out, bool* empty) {
  *empty = false;
  if (T < 0 || R < 0 || k < 0) return SV_ERR_SHAPE;
  if ((long long)R * (k + 1) != (long long)T) return SV_ERR_SHAPE;
  if (T == 0) {
    *empty = true;
    return SV_OK;
  }
  if (V < 1) return SV_ERR_SHAPE;
  if ((long long)V > 0x7FFFFFFFll - 32768) return SV_ERR_SHAPE;
  if (!logits || !kv_lens_in || !argmax_ids || !accepted || !next_tokens || !kv_lens_out)
    return SV_ERR_NULL;
  if (k > 0 && !draft_tokens) return SV_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(logits) & 3u) return SV_ERR_ALIGN;
  const int chunk = greedy_chunk(T, V);
  const long long nchunks = (V + (long long)chunk - 1) / chunk;
  if ((long long)T * nchunks > 0x7FFFFFFFll) return SV_ERR_SHAPE;
  return SV_OK;
}

// The launch itself, after every check has passed (workspace: zero-filled,
// 256-byte aligned, at least sv_greedy_workspace_bytes(T, V) bytes).
sv_status greedy_launch(const float* logits, int T, int V, int R, int k, const int32_t* draft_tokens,
                        const int32_t* kv_lens_in, int32_t* argmax_ids, int32_t* accepted,
                        int32_t* next_tokens, int32_t* kv_lens_out, void* workspace, cudaStream_t stream) {
  const int chunk = greedy_chunk(T, V);
  const int nchunks = (int)((V + (long long)chunk - 1) / chunk);
  const long long blocks = (long long)T * nchunks;
  const bool vec4 = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
  auto* ticket = reinterpret_cast<unsigned int*>(workspace);
  auto* row_key = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + kGreedyHeader);
  greedy_verify_kernel<<<(unsigned)blocks, kGreedyThreads, 0, stream>>>(
      logits, T, V, R, k, chunk, nchunks, vec4, draft_tokens, kv_lens_in, argmax_ids, accepted,
      next_tokens, kv_lens_out, ticket, row_key);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_LAUNCH;
}

}  // namespace
}  // namespace sv

extern "C" sv_status spec_verify_greedy(const float* logits, int T, int V, int R, int k,
                                        const int32_t* draft_tokens, const int32_t* kv_lens_in,
                                        int32_t* argmax_ids, int32_t* accepted,
                                        int32_t* next_tokens, int32_t* kv_lens_out,
                                        void* workspace, size_t workspace_bytes,
                                        sv_stream_t stream) {
  bool empty = false;
  const sv_status st = sv::greedy_check(logits, T, V, R, k, draft_tokens, kv_lens_in, argmax_ids,
                                        accepted, next_tokens, kv_lens_out, &empty);
  if (st != SV_OK || empty) return st;
  if (!workspace) return SV_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return SV_ERR_ALIGN;
  if (workspace_bytes < sv_greedy_workspace_bytes(T, V)) return SV_ERR_WORKSPACE;
  return sv::greedy_launch(logits, T, V, R, k, draft_tokens, kv_lens_in, argmax_ids, accepted,
                           next_tokens, kv_lens_out, workspace, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Allocation-free variant.
//
// Some callers cannot allocate device memory at the point where they verify:
// a serving engine that has already handed (nearly) all of HBM to its own
// KV-cache pool and forbids further cudaMalloc calls, or a plugin hosted by a
// framework that owns the device allocator.  Such a caller cannot provide the
// greedy workspace.  This entry point keeps that scratch (the ticket counter
// and the per-row argmax keys) in a fixed file-scope device array instead.
//
// Limits and sharing:
//  * The array holds kNoAllocScratchBytes (512 KiB) on every GPU that loads
//    this library, until the process exits.  A problem whose workspace
//    (sv_greedy_workspace_bytes(T, V)) is larger is rejected with
//    SV_ERR_WORKSPACE; every argument is checked before anything is
//    enqueued.
//  * Every call shares the one array: calls whose kernels could overlap on the
//    GPU (different streams without ordering, or several host threads) race
//    on it and give wrong results.  Calls issued in order on one stream are
//    fine.
//  * The first call on a device (per CUDA context) looks up the array's
//    device address (cudaGetSymbolAddress) with that device current and
//    caches it with the context; a call from another context looks it up
//    again.  Make the first call before any stream capture begins.  A
//    cudaDeviceReset of the device may keep the context handle while the
//    array moves, so this entry point must not be used on a device after the
//    process has reset it.
//  * The counter and keys must start at zero: each call clears the part it
//    uses with a cudaMemsetAsync on the same stream before the kernel runs
//    (every call also leaves them zero).
// No cudaMalloc, cudaFree or other allocating routine is called.
namespace sv {
namespace {

constexpr size_t kNoAllocScratchBytes = 512 * 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

PFN_cuCtxGetCurrent_v4000 get_ctx_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
  });
  return fn;
}

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];
CUcontext g_noalloc_ctx[64];

// Device address of g_noalloc_scratch on the current device and context
// (nullptr on failure).
void* noalloc_scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  auto ctx_fn = get_ctx_fn();
  if (!ctx_fn) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  CUcontext ctx = nullptr;
  if (ctx_fn(&ctx) != CUDA_SUCCESS) return nullptr;
  if (ctx != nullptr && g_noalloc_ptr[dev] && g_noalloc_ctx[dev] == ctx) return g_noalloc_ptr[dev];
  // first call on this device or another context: the runtime call below
  // also makes the device's primary context current when none is
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  if (ctx == nullptr && (ctx_fn(&ctx) != CUDA_SUCCESS || ctx == nullptr)) return nullptr;
  g_noalloc_ptr[dev] = p;
  g_noalloc_ctx[dev] = ctx;
  return p;
}

}  // namespace
}  // namespace sv

extern "C" sv_status spec_verify_greedy_noalloc(const float* logits, int T, int V, int R, int k,
                                                const int32_t* draft_tokens,
                                                const int32_t* kv_lens_in, int32_t* argmax_ids,
                                                int32_t* accepted, int32_t* next_tokens,
                                                int32_t* kv_lens_out, sv_stream_t stream) {
  bool empty = false;
  const sv_status st = sv::greedy_check(logits, T, V, R, k, draft_tokens, kv_lens_in, argmax_ids,
                                        accepted, next_tokens, kv_lens_out, &empty);
  if (st != SV_OK || empty) return st;
  const size_t need = sv_greedy_workspace_bytes(T, V);
  if (need > sv::kNoAllocScratchBytes) return SV_ERR_WORKSPACE;
  void* scratch = sv::noalloc_scratch_for_current_device();
  if (!scratch) return SV_ERR_DEVICE;
  const cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, need, st_) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_LAUNCH;
  }
  return sv::greedy_launch(logits, T, V, R, k, draft_tokens, kv_lens_in, argmax_ids, accepted,
                           next_tokens, kv_lens_out, scratch, st_);
}
