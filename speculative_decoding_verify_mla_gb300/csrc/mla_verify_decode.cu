// mla_verify_decode.cu - absorbed, gated NoPE MLA verify-decode attention over
// a paged bf16 latent KV cache, for sm_103a (tcgen05 + TMEM + TMA + clusters).
//
// What it computes ("M* PR #257: Kimi K3 support with DSpark speculative
// decoding", sections "Model" and "Speculative decoding"; per-token bounds,
// widened masked span and the (-inf, 0) stats identity from "TensorRT-LLM PR
// #18166: Kimi K3 DSpark speculative decoding under Helix CP", first commit
// message and Summary): for token t of request r and head h, over the latent
// rows c_j (j < kv_bounds[t]) of r's pages,
//     s_j = scale <q, c_j>,  lse = ln sum exp(s_j),  o = sum exp(s_j - lse) c_j,
// then out = sigmoid(gate) * o; a zero bound gives (lse, o) = (-inf, 0).
//
// Design (one GPU, sm_103a):
//  * Fold.  The k+1 tokens of a request times H heads are M = H (k+1) query
//    rows sharing one KV stream (row = t*H + h).  A work unit is (request,
//    128-row tile, KV split) and runs on a 2-CTA cluster.
//  * Latent split across the pair.  An fp32 128 x 512 output tile would fill
//    the whole 512-column TMEM of one SM, so CTA c of the pair owns latent
//    columns [256c, 256c + 256): its TMEM holds O[:, half c] (256 columns),
//    its half of Q as a bf16 A operand (128 columns) and two 64-column score
//    buffers.  Because K = V (absorbed MLA), the same half of each KV row
//    feeds both of its GEMMs, so each CTA streams exactly half of every
//    latent row: the pair reads the KV once.
//  * Scores.  CTA c computes the partial scores Q[:, half c] K[:, half c]^T
//    (tcgen05.mma, M=128, N=64, K=256, A from TMEM, B from swizzled SMEM);
//    the two partials are swapped through distributed shared memory and
//    added (fp32, a+b in both CTAs, so both see bit-identical scores).
//  * Softmax.  One thread per query row: scale, per-token bound mask, running
//    max with a lazy rescale (O is rescaled in TMEM only when the max grows by
//    more than 2^8), exp2, bf16 P written back into the score buffer in TMEM.
//  * P V.  tcgen05.mma M=128, N=256, K=64 with A = P from TMEM and B = the
//    same SMEM tile read MN-major (V = the latent rows).
//  * KV.  TMA tiled loads of 64 rows x 64 columns (128-byte swizzle) from a
//    2-D tensor map over the page pool; the row coordinate is page * 64, so
//    the block table is applied per tile.  4-stage ring.  Pool slack beyond
//    the tile's largest bound is zeroed in SMEM before use (0 * NaN safety).
//  * Epilogue.  One split: normalise, gate, bf16 out + lse.  Several splits:
//    fp32 partials (o/l, lse) for mla_lse_combine.
//  * Roles: warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 softmax and
//    epilogue.  Every wait is bounded; nothing traps.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "sv_ptx.cuh"

namespace sv {

cudaError_t launch_lse_combine(const float* part_o, const float* part_lse, int S, long long rows,
                               const void* gate, void* out, float* lse, cudaStream_t stream);

namespace {

constexpr int kD = SV_LATENT_DIM;
constexpr int kDHalf = kD / 2;
constexpr int kTileN = SV_PAGE_SIZE;  // KV rows per tile = one page
constexpr int kMTile = 128;           // folded query rows per unit
constexpr int kStages = 4;
constexpr int kBoxBytes = 64 * 128;            // one TMA box: 64 rows x 64 bf16
constexpr int kStageBytes = 4 * kBoxBytes;     // 64 rows x 256 bf16
constexpr int kXRowBytes = 64 * 4 + 16;        // exchanged score row, padded
constexpr int kXBufBytes = kMTile * kXRowBytes;
constexpr int kThreads = 192;
constexpr int kNumBars = 18;
constexpr uint32_t kTmemO = 0, kTmemQ = 256, kTmemS = 384, kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // in log2 units
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kSmemUsed = kStages * kStageBytes + 2 * kXBufBytes + kNumBars * 8 + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct VerifyParams {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* kv_bounds;
  const __nv_bfloat16* gate;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int32_t* status;
  long long rows_total;  // T * H
  int R, q_per_req, H, max_pages, num_pages, num_splits, n_mtiles;
  float scale_log2;  // softmax_scale * log2(e)
};

__device__ __forceinline__ int load_bound(const VerifyParams& p, int tok) {
  int b = __ldg(p.kv_bounds + tok);
  const int cap = p.max_pages * kTileN;
  if (b < 0 || b > cap) {
    if (p.status) atomicOr(p.status, SV_DEV_BAD_BOUND);
    b = b < 0 ? 0 : cap;
  }
  return b;
}

// Bounded wait taken by a whole warp; all lanes get the same answer.
template <bool kCluster>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status) {
  const bool ok = mbar_wait<kCluster>(bar, parity, abort_flag, status);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Bounded wait used only while tearing down (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

__device__ __forceinline__ float sigmoidf_(float g) { return 1.0f / (1.0f + __expf(-g)); }

__global__ void __launch_bounds__(kThreads, 1)
    mla_verify_kernel(const __grid_constant__ CUtensorMap tmap_kv, const VerifyParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* const sptr = smem_raw + (sbase - raw);
  const uint32_t stage0 = sbase;
  const uint32_t xbuf0 = sbase + kStages * kStageBytes;
  const uint32_t bar0 = xbuf0 + 2 * kXBufBytes;
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (4 + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (8 + b); };
  auto p_full = [&](int b) { return bar0 + 8u * (10 + b); };
  auto pv_done = [&](int b) { return bar0 + 8u * (12 + b); };
  auto xfull = [&](int b) { return bar0 + 8u * (14 + b); };
  const uint32_t q_ready = bar0 + 8u * 16;
  const uint32_t drain_bar = bar0 + 8u * 17;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sptr + (bar0 - sbase) + 8 * kNumBars);
  volatile int* const abort_flag =
      reinterpret_cast<volatile int*>(sptr + (bar0 - sbase) + 8 * kNumBars + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const int unit = blockIdx.x >> 1;
  const int S = p.num_splits;
  const int s_idx = unit % S;
  const int rm = unit / S;
  const int m_tile = rm % p.n_mtiles;
  const int r = rm / p.n_mtiles;
  const int Mq = p.H * p.q_per_req;

  // ---- unit geometry (every thread derives the same values)
  int maxb_req = 0;
  for (int t = 0; t < p.q_per_req; ++t) maxb_req = max(maxb_req, load_bound(p, r * p.q_per_req + t));
  const int t_first = (m_tile * kMTile) / p.H;
  const int t_last = min((m_tile * kMTile + kMTile - 1) / p.H, p.q_per_req - 1);
  int maxb_tile = 0;
  for (int t = t_first; t <= t_last; ++t)
    maxb_tile = max(maxb_tile, load_bound(p, r * p.q_per_req + t));
  const int n_r = (maxb_req + kTileN - 1) / kTileN;
  const int lo = (int)((long long)s_idx * n_r / S);
  const int hi = (int)((long long)(s_idx + 1) * n_r / S);
  const int hi_eff = min(hi, (maxb_tile + kTileN - 1) / kTileN);
  const int ntiles = max(0, hi_eff - lo);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), 128);
      mbar_init(pv_done(b), 1);
      mbar_init(xfull(b), 128);
    }
    mbar_init(q_ready, 128);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  cluster_sync();  // the peer's barriers exist before any remote arrive

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tmap_kv);
      int last_round[kStages] = {-1, -1, -1, -1};
      for (int it = 0; it < ntiles; ++it) {
        const int st = it & (kStages - 1);
        const int round = it / kStages;
        if (round > 0 && !mbar_wait<false>(kv_empty(st), (round - 1) & 1, abort_flag, p.status))
          break;
        mbar_arrive_expect_tx(kv_full(st), kStageBytes);
        const int j = lo + it;
        int page = __ldg(p.block_table + (long long)r * p.max_pages + j);
        if (page < 0 || page >= p.num_pages) {
          if (p.status) atomicOr(p.status, SV_DEV_BAD_PAGE);
          page = 0;
        }
        const uint32_t dst = stage0 + st * kStageBytes;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tma_load_2d(dst + b * kBoxBytes, &tmap_kv, kv_full(st), (int)crank * kDHalf + b * 64,
                      page * kTileN);
        last_round[st] = round;
      }
      // every copy this CTA started has landed before teardown
      for (int st = 0; st < kStages; ++st)
        if (last_round[st] >= 0) drain_wait(kv_full(st), last_round[st] & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
    bool ok = ntiles > 0 && warp_wait<false>(q_ready, 0, abort_flag, p.status);
    bool issued = false;
    auto issue_pv = [&](int i) -> bool {
      const int sb = i & 1;
      const int st = i & (kStages - 1);
      if (!warp_wait<false>(p_full(sb), (i >> 1) & 1, abort_flag, p.status)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a = tmem + kTmemS + 64u * sb;
        const uint32_t sa = stage0 + st * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // B = V tile, MN-major: N = 256 latent columns in four 64-wide boxes
          // (LBO = box stride), K = 16 KV rows per step (SBO = 8-row stride).
          const uint64_t bd = sdesc_sw128(sa + kk * 16 * 128, kBoxBytes, 1024);
          mma_ts(tmem + kTmemO, a + 8u * kk, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(kv_empty(st));
        mma_commit(pv_done(sb));
      }
      __syncwarp();
      return true;
    };
    if (ok) tc_fence_after();
    for (int it = 0; ok && it < ntiles; ++it) {
      const int st = it & (kStages - 1);
      const int sb = it & 1;
      if (!warp_wait<false>(kv_full(st), (it / kStages) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const int rows_valid = maxb_tile - (lo + it) * kTileN;
      if (rows_valid < kTileN) {
        // rows no query row of this tile may see: zero them (pool slack may be NaN)
        uint8_t* tile = sptr + (stage0 - sbase) + st * kStageBytes;
        const int nrows = kTileN - rows_valid;
        for (int idx = lane; idx < nrows * 4 * 8; idx += 32) {
          const int c16 = idx & 7;
          const int rr = (idx >> 3) % nrows;
          const int b = (idx >> 3) / nrows;
          *reinterpret_cast<uint4*>(tile + b * kBoxBytes + (rows_valid + rr) * 128 + c16 * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sa = stage0 + st * kStageBytes;
        const uint32_t d = tmem + kTmemS + 64u * sb;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          // B = K tile, K-major, 128-byte swizzle: step 16 latent columns
          // (32 bytes) inside a box, next box every 4 steps.
          const uint64_t bd = sdesc_sw128(sa + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024);
          mma_ts(d, tmem + kTmemQ + 8u * kk, bd, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full(sb));
      }
      __syncwarp();
      issued = true;
      if (it >= 1 && !issue_pv(it - 1)) {
        ok = false;
        break;
      }
    }
    if (ok && ntiles > 0) ok = issue_pv(ntiles - 1);
    if (issued && lane == 0) {
      mma_commit(drain_bar);
      drain_wait(drain_bar, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int wq = warp & 3;  // TMEM lane quadrant of this warp
    const int i = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int f = m_tile * kMTile + i;
    const bool valid = f < Mq;
    const int t_loc = valid ? f / p.H : 0;
    const long long row_g = (long long)r * Mq + f;
    const int b_i = valid ? load_bound(p, r * p.q_per_req + t_loc) : 0;

    if (ntiles > 0) {
      // this CTA's half of the query row -> TMEM (bf16 pairs per 32-bit column)
      const uint4* src = reinterpret_cast<const uint4*>(p.q + row_g * kD + crank * kDHalf);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = valid ? __ldg(src + c * 8 + u) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * u + 0] = x.x;
          v[4 * u + 1] = x.y;
          v[4 * u + 2] = x.z;
          v[4 * u + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + kTmemQ + 32u * c, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
    }

    float m_ref = -INFINITY;  // running max (log2 units) used for exponentiation
    float l_sum = 0.f;
    const uint32_t my_x = xbuf0 + (uint32_t)i * kXRowBytes;
    const uint32_t peer_x = mapa_shared(my_x, peer);
    const uint32_t peer_xfull0 = mapa_shared(xfull(0), peer);
    const uint32_t peer_xfull1 = mapa_shared(xfull(1), peer);
    bool ok = true;
    for (int it = 0; it < ntiles; ++it) {
      const int sb = it & 1;
      const uint32_t par = (it >> 1) & 1;
      if (!warp_wait<false>(s_full(sb), par, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      float x[64];
      {
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_off + kTmemS + 64u * sb, a);
        tmem_ld32(tmem + lane_off + kTmemS + 64u * sb + 32u, b);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(a[c]);
          x[32 + c] = __uint_as_float(b[c]);
        }
      }
      // swap partial scores with the peer CTA (other latent half)
      const uint32_t dst = peer_x + (uint32_t)sb * kXBufBytes;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_cluster_v4(dst + 16u * c, x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
      mbar_arrive_cluster(sb ? peer_xfull1 : peer_xfull0);
      if (!warp_wait<true>(xfull(sb), par, abort_flag, p.status)) { ok = false; break; }
      const float4* theirs =
          reinterpret_cast<const float4*>(sptr + (my_x - sbase) + (uint32_t)sb * kXBufBytes);
      const int lim = b_i - (lo + it) * kTileN;  // columns >= lim are masked
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float4 y = theirs[c];
        float v0 = (x[4 * c + 0] + y.x) * p.scale_log2;
        float v1 = (x[4 * c + 1] + y.y) * p.scale_log2;
        float v2 = (x[4 * c + 2] + y.z) * p.scale_log2;
        float v3 = (x[4 * c + 3] + y.w) * p.scale_log2;
        if (4 * c + 0 >= lim) v0 = -INFINITY;
        if (4 * c + 1 >= lim) v1 = -INFINITY;
        if (4 * c + 2 >= lim) v2 = -INFINITY;
        if (4 * c + 3 >= lim) v3 = -INFINITY;
        x[4 * c + 0] = v0;
        x[4 * c + 1] = v1;
        x[4 * c + 2] = v2;
        x[4 * c + 3] = v3;
        tmax = fmaxf(tmax, fmaxf(fmaxf(v0, v1), fmaxf(v2, v3)));
      }
      // lazy rescale: move the reference max only when it grows by > 2^8
      const bool move = tmax > m_ref + kRescaleThreshold;
      const float m_new = move ? tmax : m_ref;
      const bool rescale_o = move && (m_ref != -INFINITY);
      const float alpha = rescale_o ? exp2f(m_ref - m_new) : 1.0f;
      if (__any_sync(0xFFFFFFFFu, rescale_o)) {
        // O holds tiles < it: wait for PV(it-1), then scale the row in TMEM
        if (!warp_wait<false>(pv_done((it - 1) & 1), ((it - 1) >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + kTmemO + 32u * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) * alpha);
          tmem_st32(tmem + lane_off + kTmemO + 32u * c, v);
        }
        tmem_wait_st();
      }
      l_sum *= alpha;
      m_ref = m_new;
      const float msub = (m_ref == -INFINITY) ? 0.f : m_ref;
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = exp2f(x[2 * c] - msub);
        const float p1 = exp2f(x[2 * c + 1] - msub);
        psum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l_sum += psum;
      tmem_st32(tmem + lane_off + kTmemS + 64u * sb, pk);  // P over the consumed scores
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full(sb));
    }

    // ---- epilogue
    if (ok && ntiles > 0)
      ok = warp_wait<false>(pv_done((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1, abort_flag,
                            p.status);
    tc_fence_after();
    const bool have_o = ok && ntiles > 0;
    const float inv_l = (l_sum > 0.f) ? 1.0f / l_sum : 0.f;
    const float lse_v = (l_sum > 0.f) ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
    if (S == 1) {
      const uint4* g = reinterpret_cast<const uint4*>(p.gate + row_g * kD + crank * kDHalf);
      uint4* o = reinterpret_cast<uint4*>(p.out + row_g * kD + crank * kDHalf);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        if (have_o) {
          tmem_ld32(tmem + lane_off + kTmemO + 32u * c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 graw = __ldg(g + 4 * c + u);
            const uint32_t gw[4] = {graw.x, graw.y, graw.z, graw.w};
            uint32_t ow[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
              const float o0 = __uint_as_float(v[8 * u + 2 * e]) * inv_l * sigmoidf_(gf.x);
              const float o1 = __uint_as_float(v[8 * u + 2 * e + 1]) * inv_l * sigmoidf_(gf.y);
              ow[e] = pack_bf16x2(o0, o1);
            }
            o[4 * c + u] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
          }
        }
      }
      if (valid && crank == 0) p.lse[row_g] = lse_v;
    } else {
      float4* po = reinterpret_cast<float4*>(p.part_o + ((long long)s_idx * p.rows_total + row_g) * kD +
                                             crank * kDHalf);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        if (have_o) {
          tmem_ld32(tmem + lane_off + kTmemO + 32u * c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            po[8 * c + u] = make_float4(__uint_as_float(v[4 * u]) * inv_l,
                                        __uint_as_float(v[4 * u + 1]) * inv_l,
                                        __uint_as_float(v[4 * u + 2]) * inv_l,
                                        __uint_as_float(v[4 * u + 3]) * inv_l);
        }
      }
      if (valid && crank == 0) p.part_lse[(long long)s_idx * p.rows_total + row_g] = lse_v;
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // neither CTA leaves while the peer may still touch its SMEM
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
bool g_attr_set[kMaxDevices];
std::mutex g_dev_mu;

bool device_setup(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_attr_set[dev]) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaFuncSetAttribute(mla_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return false;
    g_sm_count[dev] = sms;
    g_attr_set[dev] = true;
  }
  if (sm_count) *sm_count = g_sm_count[dev];
  return true;
}

int auto_splits(int R, int q_per_req, int H, int max_pages, int sm_count) {
  const long long n_mt = ((long long)H * q_per_req + kMTile - 1) / kMTile;
  const long long pairs = (long long)R * n_mt;
  if (pairs <= 0) return 1;
  long long s = (long long)sm_count / (2 * pairs);
  const long long by_len = max_pages / 4;
  if (s > by_len) s = by_len;
  if (s > SV_MAX_SPLITS) s = SV_MAX_SPLITS;
  if (s < 1) s = 1;
  return (int)s;
}

inline bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

}  // namespace
}  // namespace sv

extern "C" int sv_mla_verify_num_splits(int R, int q_per_req, int H, int max_pages_per_req) {
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
  }
  return sv::auto_splits(R, q_per_req, H, max_pages_per_req, sms);
}

extern "C" size_t sv_mla_verify_workspace_bytes(int T, int H, int num_splits) {
  if (T <= 0 || H <= 0 || num_splits <= 1) return 0;
  const size_t rows = (size_t)T * (size_t)H;
  const size_t o_bytes = (size_t)num_splits * rows * sv::kD * sizeof(float);
  return o_bytes + (size_t)num_splits * rows * sizeof(float);
}

extern "C" sv_status mla_verify_decode(const void* q_latent, const void* kv_pages, int num_pages,
                                       int page_size, const int32_t* block_table, int R,
                                       int q_per_req, int max_pages_per_req,
                                       const int32_t* kv_bounds, const void* gate, int H,
                                       float softmax_scale, int num_splits, void* workspace,
                                       size_t workspace_bytes, void* out, float* lse,
                                       int32_t* status, sv_stream_t stream) {
  using namespace sv;
  if (R < 0 || q_per_req < 1 || H < 1 || max_pages_per_req < 0 || num_pages < 0)
    return SV_ERR_SHAPE;
  if (page_size != SV_PAGE_SIZE) return SV_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > SV_MAX_SPLITS) return SV_ERR_SHAPE;
  const long long T = (long long)R * q_per_req;
  if (T == 0) return SV_OK;
  if (T * H > (1ll << 40) || (long long)num_pages * kTileN > 0x7FFFFFFFll) return SV_ERR_SHAPE;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return SV_ERR_SHAPE;
  if (num_pages < 1 || max_pages_per_req < 1) return SV_ERR_SHAPE;
  if (!q_latent || !kv_pages || !block_table || !kv_bounds || !gate || !out || !lse)
    return SV_ERR_NULL;
  if (misaligned(q_latent, 16) || misaligned(kv_pages, 16) || misaligned(gate, 16) ||
      misaligned(out, 16) || misaligned(lse, 4) || misaligned(block_table, 4) ||
      misaligned(kv_bounds, 4))
    return SV_ERR_ALIGN;
  int sm_count = 0;
  if (!device_setup(&sm_count)) return SV_ERR_DEVICE;
  const int S = num_splits > 0 ? num_splits
                               : auto_splits(R, q_per_req, H, max_pages_per_req, sm_count);
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (S > 1) {
    if (!workspace) return SV_ERR_WORKSPACE;
    if (misaligned(workspace, 256)) return SV_ERR_ALIGN;
    if (workspace_bytes < sv_mla_verify_workspace_bytes((int)T, H, S)) return SV_ERR_WORKSPACE;
    part_o = static_cast<float*>(workspace);
    part_lse = part_o + (size_t)S * T * H * kD;
  }
  auto encode = get_encode_fn();
  if (!encode) return SV_ERR_DEVICE;
  CUtensorMap tmap;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)num_pages * kTileN};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_pages), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return SV_ERR_ALIGN;

  VerifyParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q_latent);
  prm.block_table = block_table;
  prm.kv_bounds = kv_bounds;
  prm.gate = static_cast<const __nv_bfloat16*>(gate);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.part_o = part_o;
  prm.part_lse = part_lse;
  prm.status = status;
  prm.rows_total = T * H;
  prm.R = R;
  prm.q_per_req = q_per_req;
  prm.H = H;
  prm.max_pages = max_pages_per_req;
  prm.num_pages = num_pages;
  prm.num_splits = S;
  prm.n_mtiles = (int)(((long long)H * q_per_req + kMTile - 1) / kMTile);
  prm.scale_log2 = softmax_scale * 1.4426950408889634f;

  const long long units = (long long)R * prm.n_mtiles * S;
  if (2 * units > 0x7FFFFFFFll) return SV_ERR_SHAPE;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * units), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mla_verify_kernel, tmap, prm) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_LAUNCH;
  }
  if (S > 1) {
    if (launch_lse_combine(part_o, part_lse, S, T * H, gate, out, lse,
                           reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SV_ERR_LAUNCH;
  }
  return SV_OK;
}

extern "C" const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_NULL: return "null pointer";
    case SV_ERR_SHAPE: return "bad shape or size";
    case SV_ERR_ALIGN: return "misaligned pointer";
    case SV_ERR_WORKSPACE: return "workspace missing or too small";
    case SV_ERR_UNSUPPORTED: return "unsupported configuration";
    case SV_ERR_LAUNCH: return "kernel launch failed";
    case SV_ERR_DEVICE_DATA: return "bad device data";
    case SV_ERR_TIMEOUT: return "in-kernel wait timed out";
    case SV_ERR_DEVICE: return "no usable device";
  }
  return "unknown status";
}
