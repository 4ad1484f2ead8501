// spec_verify_sampled.cu - sampled (rejection-sampling) verification of
// drafted tokens with KV trim.
//
// Definition ("M* PR #257: Kimi K3 support with DSpark speculative decoding",
// section "Speculative decoding": verification is greedy or sampled, the
// sampled form being FlashInfer's chain sampling; the pages give no formula,
// so this is the token-wise chain rejection sampling of the published
// speculative sampling method, Leviathan et al. 2023 / Chen et al. 2023):
//   p_t = softmax(logits[t] / temperature);
//   draft j of request r (drawn from q_{r,j} = draft_probs[r][j]) is accepted
//   iff u[r][j] * q_{r,j}(d) < p_t(d), t = r (k+1) + j;
//   at the first rejection the next token is drawn from max(0, p_t - q_{r,j})
//   (p_t itself if that is zero everywhere); after k acceptances it is drawn
//   from p of the last verify token; a draw from weights w with uniform
//   u = u[r][k] is the smallest v with sum_{i<=v} w_i > u * sum(w);
//   kv_lens_out = kv_lens_in - (k - n).
//
// Two launches, both HBM-bound streams over fp32 rows:
//  1. sampled_stats_kernel: every (row, chunk) CTA reduces its chunk of the
//     logits to (max, sum 2^(y - max)) with y = x * log2(e) / temperature.
//     The CTA taking the last ticket merges the chunk statistics per row,
//     takes the acceptance decisions of every request (scalar reads of
//     p_t(d) and q(d)), writes accepted / kv_lens_out and, per request, the
//     row and weight kind the next token is drawn from; it resets the ticket.
//  2. sampled_draw_kernel (programmatic dependent launch): every (request,
//     chunk) CTA computes its chunk's weight total with a fixed-order tile
//     scan.  The last CTA of a request walks the chunk totals to the chunk
//     that holds u * W and rescans it with the same tile scan (so the totals
//     agree bit for bit) to find the index; it resets its ticket.
#include <cuda_runtime.h>

#include <cstdint>

#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr size_t kAlign = 256;
constexpr int kStage = 1024;  // chunk totals staged per pass in the draw kernel


struct Decision {
  int n;      // accepted drafts
  int row;    // verify token whose distribution the draw uses
  int mode;   // 0: p_row, 1: residual max(0, p_row - q_{r,n})
  int pad;
  float m2;   // row max of y (log2 domain)
  float inv_z;
  float pad2[2];
};
static_assert(sizeof(Decision) == 32, "decision record is 32 bytes");

// The decision record is written by the stats kernel, the prerequisite grid
// of the draw kernel: read it after griddepcontrol.wait with loads the
// compiler cannot hoist.
__device__ __forceinline__ Decision load_decision(const Decision* p) {
  const int4 a = ld_dep_i4(p);
  const int4 b = ld_dep_i4(reinterpret_cast<const char*>(p) + 16);
  Decision d;
  d.n = a.x;
  d.row = a.y;
  d.mode = a.z;
  d.pad = a.w;
  d.m2 = __int_as_float(b.x);
  d.inv_z = __int_as_float(b.y);
  d.pad2[0] = __int_as_float(b.z);
  d.pad2[1] = __int_as_float(b.w);
  return d;
}

__host__ __device__ inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Chunk lengths depend on the problem only, so that the workspace query and
// the launch agree.
int stats_chunk(int T, int V) {
  const long long total = (long long)T * V;
  long long c = (total + 4 * 152 - 1) / (4 * 152);  // about four CTAs per SM
  c = (c + 8191) / 8192 * 8192;
  if (c < 8192) c = 8192;
  if (c > 65536) c = 65536;
  return (int)c;
}
int draw_chunk(int R, int V) {
  long long want = (4 * 152 + R - 1) / R;  // CTAs per request
  long long c = ((long long)V + want - 1) / want;
  c = (c + 1023) / 1024 * 1024;             // whole 1024-element tiles
  if (c < 1024) c = 1024;
  if (c > 32768) c = 32768;
  return (int)c;
}

// Bulk path (V % 4 == 0, 16-byte aligned rows): the chunk is staged in shared
// memory, logits and draft probabilities, so at most 16384 floats; the chunk
// is 1024 * m floats with m odd, so that the per-thread segments (4 m floats,
// an odd number of 16-byte words apart) hit distinct banks.
int draw_chunk_bulk(int R, int V) {
  long long want = (4 * 152 + R - 1) / R;
  long long m = ((long long)V + want * 1024 - 1) / (want * 1024);
  if (m < 1) m = 1;
  if (m % 2 == 0) ++m;
  if (m > 15) m = 15;
  return (int)(m * 1024);
}

struct Layout {
  size_t tickets2, stats, rowstat, decisions, sums, nacc, total;
  int chunk1, nch1, chunk2, nch2;
};
Layout layout(int R, int k, int V, bool bulk) {
  Layout L;
  const int T = R * (k + 1);
  L.chunk1 = stats_chunk(T, V);
  L.nch1 = (int)((V + (long long)L.chunk1 - 1) / L.chunk1);
  L.chunk2 = bulk ? draw_chunk_bulk(R, V) : draw_chunk(R, V);
  L.nch2 = (int)((V + (long long)L.chunk2 - 1) / L.chunk2);
  L.tickets2 = kAlign;                                              // after ticket 1
  L.stats = L.tickets2 + align_up((size_t)R * sizeof(unsigned int));
  L.rowstat = L.stats + align_up((size_t)T * L.nch1 * sizeof(float2));
  L.decisions = L.rowstat + align_up((size_t)T * sizeof(float2));
  L.sums = L.decisions + align_up((size_t)R * sizeof(Decision));
  L.nacc = L.sums + align_up((size_t)R * L.nch2 * sizeof(float));
  L.total = L.nacc + align_up((size_t)R * sizeof(int));
  return L;
}

__device__ __forceinline__ float4 ld_stream_f4(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Merge of two (max, sum 2^(y - max)) pairs; an empty pair is (-inf, 0).
__device__ __forceinline__ void merge_stat(float& m, float& z, float m2, float z2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; z = z2; return; }
  const float mx = fmaxf(m, m2);
  z = z * fast_exp2(m - mx) + z2 * fast_exp2(m2 - mx);
  m = mx;
}

__device__ __forceinline__ void warp_merge_stat(float& m, float& z) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float z2 = __shfl_xor_sync(0xFFFFFFFFu, z, o);
    merge_stat(m, z, m2, z2);
  }
}

// ---------------------------------------------------------------------------
// kernel 1: row statistics, then the acceptance decisions
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
    sampled_stats_kernel(const float* __restrict__ logits, int T, int V, int R, int k, float s,
                         int chunk, int nchunks, bool vec4,
                         const int32_t* __restrict__ draft_tokens,
                         const float* __restrict__ draft_probs, const float* __restrict__ uniforms,
                         const int32_t* __restrict__ kv_lens_in, int32_t* __restrict__ accepted,
                         int32_t* __restrict__ kv_lens_out, unsigned int* __restrict__ ticket,
                         float2* __restrict__ stats, float2* rowstat,
                         Decision* __restrict__ decisions, int* n_acc) {
  // shared memory stays under 1 KB (the attention kernel leaves ~1.8 KB of
  // an SM's shared memory to kernels that run beside it)
  __shared__ float s_m[kWarps], s_z[kWarps];
  __shared__ bool s_last;
  const int tid = threadIdx.x;
  const int t = (int)(blockIdx.x / nchunks);
  const int c = (int)(blockIdx.x % nchunks);
  const long long lo = (long long)c * chunk;
  const long long hi = min((long long)V, lo + chunk);
  const float* row = logits + (long long)t * V;

  // The dependent draw kernel may be scheduled as soon as SMs free up; its
  // griddepcontrol.wait holds it until this whole grid has completed, and it
  // reads the decisions only after that wait.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  float m = -INFINITY, z = 0.f;
  if (vec4) {
    const float4* p4 = reinterpret_cast<const float4*>(row + lo);
    const int n4 = (int)((hi - lo) >> 2);
    int i = tid;
    for (; i + 7 * kThreads < n4; i += 8 * kThreads) {
      float4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = ld_stream_f4(p4 + i + u * kThreads);
      float bm = m;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        bm = fmaxf(bm, fmaxf(fmaxf(a[u].x, a[u].y), fmaxf(a[u].z, a[u].w)) * s);
      if (bm > m) { z = (m == -INFINITY) ? 0.f : z * fast_exp2(m - bm); m = bm; }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        z += fast_exp2(fmaf(a[u].x, s, -m)) + fast_exp2(fmaf(a[u].y, s, -m)) +
             fast_exp2(fmaf(a[u].z, s, -m)) + fast_exp2(fmaf(a[u].w, s, -m));
    }
    for (; i < n4; i += kThreads) {
      const float4 a = ld_stream_f4(p4 + i);
      const float bm = fmaxf(m, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)) * s);
      if (bm > m) { z = (m == -INFINITY) ? 0.f : z * fast_exp2(m - bm); m = bm; }
      z += fast_exp2(fmaf(a.x, s, -m)) + fast_exp2(fmaf(a.y, s, -m)) +
           fast_exp2(fmaf(a.z, s, -m)) + fast_exp2(fmaf(a.w, s, -m));
    }
  } else {
    for (long long i = lo + tid; i < hi; i += kThreads) {
      const float y = __ldcs(row + i) * s;
      if (y > m) { z = (m == -INFINITY) ? 0.f : z * fast_exp2(m - y); m = y; }
      z += fast_exp2(y - m);
    }
  }
  // Scaling by s > 0 preserves the max: max(x) * s == max(x * s) exactly, and
  // fmaf(x, s, -m) is the rounded y - m of the same y = x * s used above up
  // to one rounding, which the tolerance of the draw covers.
  warp_merge_stat(m, z);
  if ((tid & 31) == 0) { s_m[tid >> 5] = m; s_z[tid >> 5] = z; }
  __syncthreads();
  if (tid < 32) {
    float mm = tid < kWarps ? s_m[tid] : -INFINITY;
    float zz = tid < kWarps ? s_z[tid] : 0.f;
    warp_merge_stat(mm, zz);
    if (tid == 0) {
      stats[(long long)t * nchunks + c] = make_float2(mm, zz);
      __threadfence();
      s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
    }
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA: row statistics, then the acceptance tests.  The loads of
  // each phase are issued at once (block-strided) and the results meet in
  // workspace slots (L2 atomics), so the tail costs a few memory round trips.
  // Global writes of this block are visible to its threads after
  // __syncthreads; the reads go to L2 (.cg).
  __threadfence();
  for (int r = tid; r < R; r += kThreads) n_acc[r] = k;
  for (int tt = tid; tt < T; tt += kThreads) {
    float mm = -INFINITY, zz = 0.f;
    const float2* sr = stats + (long long)tt * nchunks;
    int j = 0;
    for (; j + 4 <= nchunks; j += 4) {
      float2 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(sr + j + u);
#pragma unroll
      for (int u = 0; u < 4; ++u) merge_stat(mm, zz, v[u].x, v[u].y);
    }
    for (; j < nchunks; ++j) {
      const float2 v = __ldcg(sr + j);
      merge_stat(mm, zz, v.x, v.y);
    }
    rowstat[tt] = make_float2(mm, 1.0f / zz);
  }
  __syncthreads();
  const long long nd = (long long)R * k;
  for (long long f = tid; f < nd; f += kThreads) {
    const int r = (int)(f / k), j = (int)(f % k);
    const int t = r * (k + 1) + j;
    const int d = __ldg(draft_tokens + f);
    bool reject = true;  // a draft id outside the vocabulary is rejected (never read)
    if (d >= 0 && d < V) {
      const float2 st = __ldcg(rowstat + t);
      const float p = fast_exp2(fmaf(__ldg(logits + (long long)t * V + d), s, -st.x)) * st.y;
      const float q = __ldg(draft_probs + f * V + d);
      const float u = __ldg(uniforms + (long long)r * (k + 1) + j);
      reject = !(u * q < p);
    }
    if (reject) atomicMin(n_acc + r, j);
  }
  __syncthreads();
  for (int r = tid; r < R; r += kThreads) {
    const int n = __ldcg(n_acc + r);
    const int base = r * (k + 1);
    Decision dcs;
    dcs.n = n;
    dcs.row = base + n;
    dcs.mode = n < k ? 1 : 0;
    dcs.pad = 0;
    const float2 st = __ldcg(rowstat + base + n);
    dcs.m2 = st.x;
    dcs.inv_z = st.y;
    dcs.pad2[0] = dcs.pad2[1] = 0.f;
    decisions[r] = dcs;
    accepted[r] = n;
    kv_lens_out[r] = kv_lens_in[r] - (k - n);
  }
  if (tid == 0) *ticket = 0u;
}

// ---------------------------------------------------------------------------
// kernel 2: weight totals per chunk, then the inverse-CDF draw
// ---------------------------------------------------------------------------
// Fixed-order block scan of one value per thread: returns the exclusive prefix
// of this thread within the tile and the tile total (identical on every call
// with the same inputs).
__device__ __forceinline__ void block_scan(float v, float& excl, float& total, float* s_w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  float ex = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (lane == 0) ex = 0.f;
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    float w = lane < kWarps ? s_w[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) s_w[kWarps + lane] = w;
  }
  __syncthreads();
  excl = (warp > 0 ? s_w[kWarps + warp - 1] : 0.f) + ex;
  total = s_w[2 * kWarps - 1];
  __syncthreads();
}

// Weight of vocabulary id v of the draw row.
__device__ __forceinline__ float draw_weight(float x, float q, float s, float m2, float inv_z,
                                             bool residual) {
  const float p = fast_exp2(fmaf(x, s, -m2)) * inv_z;
  return residual ? fmaxf(p - q, 0.f) : p;
}

// Scan of [lo, hi) of the draw row in 1024-element tiles (four consecutive ids
// per thread), tiles taken in increasing order.  The loads of up to kBatch
// tiles are issued before the first of their scans, so that one CTA keeps
// several tiles in flight; the arithmetic and its order do not depend on the
// batching, so every call over the same range gives the same running sums.
// Returns the total; with search, also the first id whose running sum exceeds
// `target` (-1 if none does).
constexpr int kBatch = 8;

template <bool kVec>
__device__ float chunk_scan(const float* __restrict__ xr, const float* __restrict__ qr,
                            long long lo, long long hi, float s, float m2, float inv_z,
                            bool residual, bool search, float target, int* s_found,
                            int* found, float* s_w) {
  float run = 0.f;
  if (search && threadIdx.x == 0) *s_found = 0x7FFFFFFF;
  __syncthreads();
  bool done = false;
  for (long long b0 = lo; b0 < hi && !done; b0 += (long long)kBatch * 4 * kThreads) {
    float4 xb[kBatch], qb[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const long long i = b0 + (long long)u * 4 * kThreads + 4ll * threadIdx.x;
      xb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      qb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kVec && i + 3 < hi) {
        xb[u] = __ldcg(reinterpret_cast<const float4*>(xr + i));
        if (residual) qb[u] = __ldcg(reinterpret_cast<const float4*>(qr + i));
      } else if (i < hi) {
        float* xs = &xb[u].x;
        float* qs = &qb[u].x;
        for (int e = 0; e < 4; ++e)
          if (i + e < hi) {
            xs[e] = __ldcg(xr + i + e);
            if (residual) qs[e] = __ldcg(qr + i + e);
          }
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const long long t0 = b0 + (long long)u * 4 * kThreads;
      if (t0 >= hi) break;  // uniform across the block
      const long long i = t0 + 4ll * threadIdx.x;
      float w[4];
      const float* xs = &xb[u].x;
      const float* qs = &qb[u].x;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = (i + e < hi) ? draw_weight(xs[e], qs[e], s, m2, inv_z, residual) : 0.f;
      const float mine = ((w[0] + w[1]) + w[2]) + w[3];
      float excl, total;
      block_scan(mine, excl, total, s_w);
      if (search) {
        float acc = run + excl;
        for (int e = 0; e < 4; ++e) {
          acc += w[e];
          if (w[e] > 0.f && acc > target) { atomicMin(s_found, (int)(i + e)); break; }
        }
        __syncthreads();
        if (*s_found != 0x7FFFFFFF) { done = true; break; }
      }
      run += total;
    }
  }
  if (search) {
    __syncthreads();
    *found = *s_found == 0x7FFFFFFF ? -1 : *s_found;
  }
  return run;
}

// Largest id in [lo, hi) with positive weight (-1 if none): the draw when
// rounding leaves u * W at or above the last running sum.
__device__ int last_positive(const float* __restrict__ xr, const float* __restrict__ qr,
                             long long lo, long long hi, float s, float m2, float inv_z,
                             bool residual, int* s_idx) {
  if (threadIdx.x == 0) *s_idx = -1;
  __syncthreads();
  int best = -1;
  for (long long i = lo + threadIdx.x; i < hi; i += kThreads) {
    const float w = draw_weight(__ldcg(xr + i), residual ? __ldcg(qr + i) : 0.f, s, m2, inv_z,
                                residual);
    if (w > 0.f) best = (int)i;
  }
  if (best >= 0) atomicMax(s_idx, best);
  __syncthreads();
  const int r = *s_idx;
  __syncthreads();
  return r;
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads)
    sampled_draw_kernel(const float* __restrict__ logits, int V, int R, int k, float s,
                        int chunk, int nchunks, const float* __restrict__ draft_probs,
                        const float* __restrict__ uniforms, int32_t* __restrict__ next_tokens,
                        unsigned int* __restrict__ tickets, const Decision* decisions,
                        float* __restrict__ sums) {
  __shared__ float s_w[2 * kWarps];
  __shared__ float s_stage[kStage];
  __shared__ float s_total, s_local_target;
  __shared__ int s_found, s_chunk, s_clamped;
  __shared__ bool s_last;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int r = (int)(blockIdx.x / nchunks);
  const int c = (int)(blockIdx.x % nchunks);
  const Decision d = load_decision(decisions + r);
  bool residual = d.mode == 1;
  const float* xr = logits + (long long)d.row * V;
  const float* qr = residual ? draft_probs + ((long long)r * k + d.n) * V : xr;
  const long long lo = (long long)c * chunk;
  const long long hi = min((long long)V, lo + chunk);
  int dummy;
  const float tot = chunk_scan<kVec>(xr, qr, lo, hi, s, d.m2, d.inv_z, residual, false, 0.f,
                                     &s_found, &dummy, s_w);
  if (threadIdx.x == 0) {
    sums[(long long)r * nchunks + c] = tot;
    __threadfence();
    s_last = (atomicAdd(tickets + r, 1u) == (unsigned)nchunks - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of request r: locate the chunk, then the id
  __threadfence();
  const float u = __ldg(uniforms + (long long)r * (k + 1) + k);
  // The chunk totals are staged in shared memory (all threads load, one
  // thread adds them in chunk order), first for W, then for the chunk whose
  // running sum first exceeds u * W (the same sums in the same order).
  const float* rs = sums + (long long)r * nchunks;
  float W_acc = 0.f;
  for (int b0 = 0; b0 < nchunks; b0 += kStage) {
    const int nb = min(kStage, nchunks - b0);
    for (int j = threadIdx.x; j < nb; j += kThreads) s_stage[j] = __ldcg(rs + b0 + j);
    __syncthreads();
    if (threadIdx.x == 0)
      for (int j = 0; j < nb; ++j) W_acc += s_stage[j];
    __syncthreads();
  }
  if (threadIdx.x == 0) s_total = W_acc;
  __syncthreads();
  {
    const float target = u * s_total;
    float cum = 0.f, before = 0.f;
    int cs = -1, last_pos = -1;
    for (int b0 = 0; b0 < nchunks; b0 += kStage) {
      const int nb = min(kStage, nchunks - b0);
      for (int j = threadIdx.x; j < nb; j += kThreads) s_stage[j] = __ldcg(rs + b0 + j);
      __syncthreads();
      if (threadIdx.x == 0) {
        for (int j = 0; j < nb; ++j) {
          const float sj = s_stage[j];
          if (sj > 0.f) last_pos = b0 + j;
          const float nc = cum + sj;
          if (cs < 0 && nc > target) { cs = b0 + j; before = cum; }
          cum = nc;
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      int clamped = 0;
      if (cs < 0) {  // u * W rounded up to W: the draw is the last positive id
        clamped = 1;
        cs = last_pos >= 0 ? last_pos : nchunks - 1;
      }
      s_chunk = cs;
      s_clamped = clamped;
      s_local_target = target - before;
    }
  }
  __syncthreads();
  const float W = s_total;
  int pick = -1;
  if (W > 0.f) {
    const int cs = s_chunk;
    const float lt = s_local_target;
    const long long slo = (long long)cs * chunk;
    const long long shi = min((long long)V, slo + chunk);
    if (!s_clamped)
      chunk_scan<kVec>(xr, qr, slo, shi, s, d.m2, d.inv_z, residual, true, lt, &s_found, &pick,
                       s_w);
    if (pick < 0) pick = last_positive(xr, qr, slo, shi, s, d.m2, d.inv_z, residual, &s_found);
  } else {
    // residual zero everywhere: draw from p of the same row over the whole row
    residual = false;
    const float Wp = chunk_scan<kVec>(xr, qr, 0, V, s, d.m2, d.inv_z, false, false, 0.f,
                                      &s_found, &dummy, s_w);
    chunk_scan<kVec>(xr, qr, 0, V, s, d.m2, d.inv_z, false, true, u * Wp, &s_found, &pick, s_w);
    if (pick < 0) pick = last_positive(xr, qr, 0, V, s, d.m2, d.inv_z, false, &s_found);
  }
  if (threadIdx.x == 0) {
    next_tokens[r] = pick < 0 ? 0 : pick;
    tickets[r] = 0u;
  }
}

// ---------------------------------------------------------------------------
// kernel 2, bulk path: the CTA's chunk of the draw row (and of the draft row
// in residual mode) arrives in shared memory by one TMA bulk copy each; every
// thread sums one contiguous segment in id order and a single block scan
// orders the segments.  The rescan of the crossing chunk repeats exactly the
// same arithmetic on the same bytes.
// ---------------------------------------------------------------------------
struct BulkCtx {
  float* sx;   // [chunk] logits of the draw row
  float* sq;   // [chunk] draft probabilities (residual mode)
  uint32_t bar;
  uint32_t phase;
  volatile int* abort_flag;
};

// Copy [lo, lo + n) of the draw row (and draft row) into shared memory and
// wait for it.  Returns false when the wait gave up.
__device__ bool bulk_stage(BulkCtx& cx, const float* xr, const float* qr, long long lo, int n,
                           bool residual) {
  __syncthreads();  // nobody still reads the previous contents
  if (threadIdx.x == 0) {
    fence_proxy_async_smem();
    const uint32_t bytes = (uint32_t)n * 4u;
    mbar_arrive_expect_tx(cx.bar, residual ? 2u * bytes : bytes);
    bulk_load(smem_u32(cx.sx), xr + lo, bytes, cx.bar);
    if (residual) bulk_load(smem_u32(cx.sq), qr + lo, bytes, cx.bar);
  }
  const bool ok = mbar_wait<false>(cx.bar, cx.phase, cx.abort_flag, nullptr);
  cx.phase ^= 1u;
  __syncthreads();
  return ok && !*cx.abort_flag;
}

// Segment sums + one block scan over the staged chunk of n ids starting at
// row id lo.  Returns the chunk total; with search, the first id whose running
// sum exceeds `target` (local to the chunk), else -1.
__device__ float bulk_scan(const BulkCtx& cx, long long lo, int n, float s, float m2, float inv_z,
                           bool residual, bool search, float target, int* s_found, float* s_w,
                           int* found) {
  const int seg = (n + 4 * kThreads - 1) / (4 * kThreads) * 4;  // ids per thread, multiple of 4
  const int b = min(n, (int)threadIdx.x * seg);
  const int e = min(n, b + seg);
  float acc = 0.f;
  for (int i = b; i < e; i += 4) {
    const float4 x4 = *reinterpret_cast<const float4*>(cx.sx + i);
    const float4 q4 = residual ? *reinterpret_cast<const float4*>(cx.sq + i)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    acc += draw_weight(x4.x, q4.x, s, m2, inv_z, residual);
    acc += draw_weight(x4.y, q4.y, s, m2, inv_z, residual);
    acc += draw_weight(x4.z, q4.z, s, m2, inv_z, residual);
    acc += draw_weight(x4.w, q4.w, s, m2, inv_z, residual);
  }
  if (search && threadIdx.x == 0) *s_found = 0x7FFFFFFF;
  float excl, total;
  block_scan(acc, excl, total, s_w);  // its barriers also publish *s_found
  if (search) {
    if (acc > 0.f && excl <= target && target < excl + acc) {
      const float lt = target - excl;
      float a = 0.f;
      for (int i = b; i < e; ++i) {
        const float w = draw_weight(cx.sx[i], residual ? cx.sq[i] : 0.f, s, m2, inv_z, residual);
        a += w;
        if (w > 0.f && a > lt) { atomicMin(s_found, (int)(lo + i)); break; }
      }
    }
    __syncthreads();
    *found = *s_found == 0x7FFFFFFF ? -1 : *s_found;
    __syncthreads();
  }
  return total;
}

// Largest id of the staged chunk with positive weight (-1 if none).
__device__ int bulk_last_positive(const BulkCtx& cx, long long lo, int n, float s, float m2,
                                  float inv_z, bool residual, int* s_idx) {
  if (threadIdx.x == 0) *s_idx = -1;
  __syncthreads();
  int best = -1;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const float w = draw_weight(cx.sx[i], residual ? cx.sq[i] : 0.f, s, m2, inv_z, residual);
    if (w > 0.f) best = (int)(lo + i);
  }
  if (best >= 0) atomicMax(s_idx, best);
  __syncthreads();
  const int r = *s_idx;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads)
    sampled_draw_bulk_kernel(const float* __restrict__ logits, int V, int R, int k, float s,
                             int chunk, int nchunks, const float* __restrict__ draft_probs,
                             const float* __restrict__ uniforms, int32_t* __restrict__ next_tokens,
                             unsigned int* __restrict__ tickets,
                             const Decision* decisions, float* __restrict__ sums) {
  extern __shared__ __align__(128) float s_buf[];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ float s_w[2 * kWarps];
  __shared__ float s_stage[kStage];
  __shared__ float s_total, s_local_target;
  __shared__ int s_found, s_chunk, s_clamped, s_abort;
  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&s_bar), 1);
    fence_mbar_init_cluster();
    s_abort = 0;
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  BulkCtx cx{s_buf, s_buf + chunk, smem_u32(&s_bar), 0u, &s_abort};
  const int r = (int)(blockIdx.x / nchunks);
  const int c = (int)(blockIdx.x % nchunks);
  const Decision d = load_decision(decisions + r);
  bool residual = d.mode == 1;
  const float* xr = logits + (long long)d.row * V;
  const float* qr = residual ? draft_probs + ((long long)r * k + d.n) * V : xr;
  const long long lo = (long long)c * chunk;
  const int n = (int)min((long long)chunk, (long long)V - lo);
  int dummy;
  if (!bulk_stage(cx, xr, qr, lo, n, residual)) {
    if (threadIdx.x == 0) next_tokens[r] = -1;
    return;
  }
  const float tot = bulk_scan(cx, lo, n, s, d.m2, d.inv_z, residual, false, 0.f, &s_found, s_w,
                              &dummy);
  if (threadIdx.x == 0) {
    sums[(long long)r * nchunks + c] = tot;
    __threadfence();
    s_last = (atomicAdd(tickets + r, 1u) == (unsigned)nchunks - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of request r: W, the crossing chunk, then the id
  __threadfence();
  const float u = __ldg(uniforms + (long long)r * (k + 1) + k);
  const float* rs = sums + (long long)r * nchunks;
  if (nchunks <= kStage) {
    // one staging: running sums in place (chunk order, one thread), then the
    // first running sum above u * W found by all threads at once
    for (int j = threadIdx.x; j < nchunks; j += kThreads) s_stage[j] = __ldcg(rs + j);
    __syncthreads();
    if (threadIdx.x == 0) {
      float cum = 0.f;
      for (int j = 0; j < nchunks; ++j) { cum += s_stage[j]; s_stage[j] = cum; }
      s_total = cum;
      s_chunk = -1;
    }
    __syncthreads();
    const float target = u * s_total;
    for (int j = threadIdx.x; j < nchunks; j += kThreads) {
      const float before = j > 0 ? s_stage[j - 1] : 0.f;
      if (s_stage[j] > target && before <= target) {
        s_chunk = j;  // unique: the running sums never decrease
        s_local_target = target - before;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_chunk < 0) {  // u * W rounded up to W
      int cs = nchunks - 1;
      while (cs > 0 && !(s_stage[cs] > (cs > 0 ? s_stage[cs - 1] : 0.f))) --cs;
      s_chunk = cs;
      s_clamped = 1;
    } else if (threadIdx.x == 0) {
      s_clamped = 0;
    }
    __syncthreads();
  } else {
  float W_acc = 0.f;
  for (int b0 = 0; b0 < nchunks; b0 += kStage) {
    const int nb = min(kStage, nchunks - b0);
    for (int j = threadIdx.x; j < nb; j += kThreads) s_stage[j] = __ldcg(rs + b0 + j);
    __syncthreads();
    if (threadIdx.x == 0)
      for (int j = 0; j < nb; ++j) W_acc += s_stage[j];
    __syncthreads();
  }
  if (threadIdx.x == 0) s_total = W_acc;
  __syncthreads();
  {
    const float target = u * s_total;
    float cum = 0.f, before = 0.f;
    int cs = -1, last_pos = -1;
    for (int b0 = 0; b0 < nchunks; b0 += kStage) {
      const int nb = min(kStage, nchunks - b0);
      for (int j = threadIdx.x; j < nb; j += kThreads) s_stage[j] = __ldcg(rs + b0 + j);
      __syncthreads();
      if (threadIdx.x == 0) {
        for (int j = 0; j < nb; ++j) {
          const float sj = s_stage[j];
          if (sj > 0.f) last_pos = b0 + j;
          const float nc = cum + sj;
          if (cs < 0 && nc > target) { cs = b0 + j; before = cum; }
          cum = nc;
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      int clamped = 0;
      if (cs < 0) {  // u * W rounded up to W: the draw is the last positive id
        clamped = 1;
        cs = last_pos >= 0 ? last_pos : nchunks - 1;
      }
      s_chunk = cs;
      s_clamped = clamped;
      s_local_target = target - before;
    }
  }
  __syncthreads();
  }
  int pick = -1;
  bool ok = true;
  if (s_total > 0.f) {
    const int cs = s_chunk;
    const long long slo = (long long)cs * chunk;
    const int sn = (int)min((long long)chunk, (long long)V - slo);
    ok = bulk_stage(cx, xr, qr, slo, sn, residual);
    if (ok) {
      if (!s_clamped)
        bulk_scan(cx, slo, sn, s, d.m2, d.inv_z, residual, true, s_local_target, &s_found, s_w,
                  &pick);
      if (pick < 0) pick = bulk_last_positive(cx, slo, sn, s, d.m2, d.inv_z, residual, &s_found);
    }
  } else {
    // residual zero everywhere: draw from p of the same row, chunk by chunk
    residual = false;
    float Wp = 0.f;
    for (int j = 0; j < nchunks && ok; ++j) {
      const long long jl = (long long)j * chunk;
      const int jn = (int)min((long long)chunk, (long long)V - jl);
      ok = bulk_stage(cx, xr, qr, jl, jn, false);
      if (ok) Wp += bulk_scan(cx, jl, jn, s, d.m2, d.inv_z, false, false, 0.f, &s_found, s_w, &dummy);
    }
    const float target = u * Wp;
    float cum = 0.f;
    int last_chunk = -1;
    for (int j = 0; j < nchunks && ok && pick < 0; ++j) {
      const long long jl = (long long)j * chunk;
      const int jn = (int)min((long long)chunk, (long long)V - jl);
      ok = bulk_stage(cx, xr, qr, jl, jn, false);
      if (!ok) break;
      const float tj = bulk_scan(cx, jl, jn, s, d.m2, d.inv_z, false, false, 0.f, &s_found, s_w,
                                 &dummy);
      if (tj > 0.f) last_chunk = j;
      if (cum + tj > target)
        bulk_scan(cx, jl, jn, s, d.m2, d.inv_z, false, true, target - cum, &s_found, s_w, &pick);
      cum += tj;
    }
    if (ok && pick < 0 && last_chunk >= 0) {
      const long long jl = (long long)last_chunk * chunk;
      const int jn = (int)min((long long)chunk, (long long)V - jl);
      ok = bulk_stage(cx, xr, qr, jl, jn, false);
      if (ok) pick = bulk_last_positive(cx, jl, jn, s, d.m2, d.inv_z, false, &s_found);
    }
  }
  if (threadIdx.x == 0) {
    next_tokens[r] = ok ? (pick < 0 ? 0 : pick) : -1;
    tickets[r] = 0u;
  }
}

}  // namespace
}  // namespace sv

extern "C" size_t sv_sampled_workspace_bytes(int R, int k, int V) {
  if (R <= 0 || k < 0 || V <= 0) return sv::kAlign;
  // the larger of the two chunkings, so that one workspace serves both paths
  const size_t a = sv::layout(R, k, V, true).total, b = sv::layout(R, k, V, false).total;
  return a > b ? a : b;
}

extern "C" sv_status spec_verify_sampled(const float* logits, int R, int k, int V,
                                         float temperature, const int32_t* draft_tokens,
                                         const float* draft_probs, const float* uniforms,
                                         const int32_t* kv_lens_in, int32_t* accepted,
                                         int32_t* next_tokens, int32_t* kv_lens_out,
                                         void* workspace, size_t workspace_bytes,
                                         sv_stream_t stream) {
  if (R < 0 || k < 0) return SV_ERR_SHAPE;
  if (R == 0) return SV_OK;
  if (V < 1 || (long long)V > 0x7FFFFFFFll - 65536) return SV_ERR_SHAPE;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return SV_ERR_SHAPE;
  const long long T = (long long)R * (k + 1);
  if (T > 0x7FFFFFFFll / 8) return SV_ERR_SHAPE;
  if (!logits || !uniforms || !kv_lens_in || !accepted || !next_tokens || !kv_lens_out ||
      !workspace)
    return SV_ERR_NULL;
  if (k > 0 && (!draft_tokens || !draft_probs)) return SV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(draft_probs) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SV_ERR_ALIGN;
  const bool vec4 = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0) &&
                    ((reinterpret_cast<uintptr_t>(draft_probs) & 15u) == 0);
  const sv::Layout L = sv::layout(R, k, V, vec4);
  if (workspace_bytes < sv_sampled_workspace_bytes(R, k, V)) return SV_ERR_WORKSPACE;
  const long long blocks1 = T * L.nch1, blocks2 = (long long)R * L.nch2;
  if (blocks1 > 0x7FFFFFFFll || blocks2 > 0x7FFFFFFFll) return SV_ERR_SHAPE;
  const float s = 1.4426950408889634f / temperature;
  char* ws = static_cast<char*>(workspace);
  auto* ticket1 = reinterpret_cast<unsigned int*>(ws);
  auto* tickets2 = reinterpret_cast<unsigned int*>(ws + L.tickets2);
  auto* stats = reinterpret_cast<float2*>(ws + L.stats);
  auto* rowstat = reinterpret_cast<float2*>(ws + L.rowstat);
  auto* dec = reinterpret_cast<sv::Decision*>(ws + L.decisions);
  auto* sums = reinterpret_cast<float*>(ws + L.sums);
  auto* nacc = reinterpret_cast<int*>(ws + L.nacc);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  sv::sampled_stats_kernel<<<(unsigned)blocks1, sv::kThreads, 0, st>>>(
      logits, (int)T, V, R, k, s, L.chunk1, L.nch1, vec4, draft_tokens, draft_probs, uniforms,
      kv_lens_in, accepted, kv_lens_out, ticket1, stats, rowstat, dec, nacc);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_LAUNCH;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks2);
  cfg.blockDim = dim3(sv::kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (vec4) {
    const size_t dyn = 2u * (size_t)L.chunk2 * sizeof(float);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
      if (cudaFuncSetAttribute(sv::sampled_draw_bulk_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               2 * 16384 * (int)sizeof(float)) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_LAUNCH;
      }
      attr_set[dev] = true;
    }
    cfg.dynamicSmemBytes = dyn;
    e = cudaLaunchKernelEx(&cfg, sv::sampled_draw_bulk_kernel, logits, V, R, k, s, L.chunk2,
                           L.nch2, draft_probs, uniforms, next_tokens, tickets2,
                           static_cast<const sv::Decision*>(dec), sums);
  } else
    e = cudaLaunchKernelEx(&cfg, sv::sampled_draw_kernel<false>, logits, V, R, k, s, L.chunk2,
                           L.nch2, draft_probs, uniforms, next_tokens, tickets2,
                           static_cast<const sv::Decision*>(dec), sums);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_LAUNCH;
  }
  return SV_OK;
}
