// mla_verify_decode.cu - absorbed, gated NoPE MLA verify-decode attention over
// a paged bf16 latent KV cache, for sm_103a (tcgen05 + TMEM + TMA).
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
//    128-row tile, KV split, latent half) and runs on one CTA.
//  * Latent halves.  An fp32 128 x 512 output tile would fill the whole
//    512-column TMEM of one SM, so a CTA owns latent columns [256c, 256c+256)
//    of O (256 TMEM columns).  Its TMEM also holds its own half of Q as a bf16
//    A operand (128 columns) and two 64-column score buffers.
//  * Scores.  The CTA computes the full 128 x 64 score tile of each 64-row KV
//    tile: Q[:, own] K[:, own]^T with A from TMEM (tcgen05.mma kind::f16,
//    M=128, N=64) plus Q[:, other] K[:, other]^T with A from swizzled SMEM.
//    Both halves of a unit therefore compute the same scores (1.5x the
//    algorithmic tensor work), but no CTA ever waits on another SM.
//  * Query.  The producer TMA-loads the CTA's query half into the idle
//    other-half KV ring and the other half into its SMEM region; the softmax
//    warps move their rows of the first into TMEM and release the ring.
//  * Softmax.  One thread per query row: scale, per-token bound mask, running
//    max with a lazy rescale (O is rescaled in TMEM only when the max grows by
//    more than 2^8), exp2, bf16 P written back into the score buffer in TMEM.
//  * P V.  tcgen05.mma M=128, N=256, K=64 with A = P from TMEM and B = the
//    own-half KV tile read MN-major (V = the latent rows, absorbed MLA).
//  * KV.  TMA tiled loads of 64 rows x 64 columns (128-byte swizzle) from a
//    2-D tensor map over the page pool; the row coordinate is page * 64, so
//    the block table is applied per tile.  The own half (used by the scores
//    and by P V) sits in a 3-stage ring; the other half (scores only) in a
//    2-stage ring that is released as soon as the score MMA completes.  Pool
//    slack beyond the tile's largest bound is zeroed in the SMEM that P V
//    reads (0 * NaN safety); in the score-only half it is masked by
//    selection.
//  * Epilogue.  One split: normalise, gate (the gate tile TMA-loaded into the
//    query region after the last score MMA), bf16 out + lse.  Several
//    splits: bf16 o/l and fp32 lse partials for the LSE merge.  The output
//    leaves in four 64-column boxes by TMA stores, each started as soon as
//    its box is staged.  In the long-unit instances four warps (one per TMEM
//    lane quadrant) are idle by then (fp8: the converters; bf16: producer
//    and MMA issuers) and take boxes 2..3 of every row.
//  * Work units.  Uniform splits decode the unit from blockIdx; the balanced
//    plan (a one-CTA plan kernel, this grid its programmatic dependent) hands
//    each CTA a unit of a list ordered longest first; the wave split mode
//    decodes it in closed form (the first k requests whole, the others in s
//    pieces, for batches between one and two waves of the SMs).
//  * MMA issue.  Separate issuing warps for the scores and for P V (and, in
//    the long-unit instances, a second score warp for the odd tiles), so
//    the tensor pipe is fed from several warps; each ring slot's descriptor
//    is built once and a K step adds a constant to its low word.
//  * Set-up.  One pass over the request's kv_bounds gives the tile's and the
//    request's KV extent (an out-of-range bound is reported once, after the
//    loads, so that they overlap).
//  * Stacked instance (M <= 64 query rows, uniform splits or the plan).  One
//    CTA holds both latent halves: rows 64..127 of its 128-row tile repeat
//    rows 0..63 (the other query half is TMA-loaded twice), so score rows L
//    and L + 64 are equal; the softmax writes P block-diagonally ([P | 0] in
//    lanes 0..63, [0 | P] in lanes 64..127) and P V runs K = 128 over the
//    tile's two latent halves, so lanes 0..63 of O accumulate latent
//    0..255 and lanes 64..127 latent 256..511.  No second CTA recomputes
//    the scores; the other-half ring is released after P V.
//  * Roles: warp 0 TMA producer, warps 2-5 softmax and epilogue, MMA
//    issuers: warp 1 the (even tiles') scores, warp 6 P V and, in the
//    long-unit instances, warp 7 the odd tiles' scores (fp8 KV: P V warp 10,
//    odd-tile warp 11; its warps 6-9 convert the KV).  Template instances:
//    KV format x one or two score warps x two-CTA or stacked form, each also
//    built with a per-launch wait limit for tests.
//    Every wait is bounded (a wait that gives up sets SV_DEV_TIMEOUT, and
//    the CTA drains what it started and frees its TMEM); nothing traps.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <array>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <utility>

#include "sv_host.h"
#include "sv_ptx.cuh"

namespace sv {

cudaError_t launch_lse_combine(const void* part_o, bool bf16_partials, const float* part_lse, int S,
                               long long rows, const void* gate, void* out, float* lse,
                               cudaStream_t stream, const int* plan_splits, const int* plan_base,
                               int Mq, int gate_dim, long long row_begin = 0, int wave_k = -1);

namespace {

constexpr int kD = SV_LATENT_DIM;
constexpr int kDHalf = kD / 2;
constexpr int kTileN = SV_PAGE_SIZE;  // KV rows per tile = one page
constexpr int kMTile = 128;           // folded query rows per unit
constexpr int kBoxBytes = 64 * 128;            // one KV TMA box: 64 rows x 64 bf16
constexpr int kHalfTileBytes = 4 * kBoxBytes;  // 64 rows x 256 bf16
constexpr int kQBoxBytes = 128 * 128;          // one Q TMA box: 128 rows x 64 bf16
constexpr int kQHalfBytes = 4 * kQBoxBytes;    // 128 rows x 256 bf16
constexpr uint32_t kEpilogueBarId = 1;  // named barrier of the softmax warps
constexpr uint32_t kHandoffBarId = 2;   // softmax warps + epilogue helper warps
constexpr uint32_t kHelperBarId = 3;    // named barrier of the epilogue helper warps
constexpr uint32_t kTmemO = 0, kTmemQ = 256, kTmemS = 384, kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // in log2 units
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kF8TileBytes = 64 * kD;  // one fp8 KV tile: 64 rows x 512 e4m3 codes
constexpr int kTwoIssuerTiles = 8;     // units with this many KV tiles use both score issuers

// Two variants of the kernel.  bf16 KV: the TMA producer fills the bf16 KV
// rings and every MMA takes bf16 operands.  fp8 KV: the MMAs take f16
// operands (e4m3 -> f16 is one exact conversion per two codes); four
// converter warps (warps 6..9) read each e4m3 tile from global memory one
// tile ahead into registers (coalesced 16-byte loads) and write it as f16
// into the same swizzled ring slots, and also write the other query half as
// f16 into shared memory; the softmax warps put their query half into TMEM
// as f16 and write P as f16.
template <bool kF8, bool kTwo>
struct KernelShape {
  static constexpr int kOwnStages = 3;
  static constexpr int kOthStages = 2;
  static constexpr int kF8Stages = 0;
  // kTwo: a second score issuer for the odd tiles (long units)
  static constexpr int kThreads = (kF8 ? 352 : 224) + (kTwo ? 32 : 0);
  static constexpr int kPvWarp = kF8 ? 10 : 6;  // issues the P V MMAs
  static constexpr int kOddWarp = kTwo ? (kF8 ? 11 : 7) : -1;  // issues the odd tiles' score MMAs
  static constexpr int kNumBars = 24;
  // Epilogue helpers of the long-unit instances: four warps, one per TMEM
  // lane quadrant, whose roles are over by the epilogue (fp8: the
  // converters; bf16: producer, score issuers and P V issuer).  They stage
  // and store output boxes 2..3 while the softmax warps do 0..1.  (The
  // short-unit fp8 instance measured slower with them: c1 23.4 -> 26.0 us.)
  static constexpr bool kHelp = kTwo;
  static constexpr int kHelperLeaderWarp = kF8 ? 6 : 0;
  __host__ __device__ static constexpr bool is_helper(int w) {
    return kTwo && (kF8 ? (w >= 6 && w < 10) : (w == 0 || w == 1 || w == 6 || w == 7));
  }
  static constexpr int kFullCount = kF8 ? 128 : 1;  // arrivals completing a KV ring slot
  // shared memory map (offsets from the 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffOwn = kOffQ + kQHalfBytes;
  static constexpr int kOffOth = kOffOwn + kOwnStages * kHalfTileBytes;
  static constexpr int kOffF8 = kOffOth + kOthStages * kHalfTileBytes;
  static constexpr int kOffBar = kOffF8 + kF8Stages * kF8TileBytes;
  static constexpr int kOffRowScale = kOffBar + kNumBars * 8 + 16;  // float[128]: 1/l per TMEM row
  static constexpr int kSmemUsed = kOffRowScale + 128 * 4;
  static constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
};
static_assert(KernelShape<false, false>::kSmemBytes == KernelShape<false, true>::kSmemBytes &&
                  KernelShape<false, false>::kSmemBytes == KernelShape<true, false>::kSmemBytes &&
                  KernelShape<false, false>::kSmemBytes == KernelShape<true, true>::kSmemBytes,
              "every instance has the same shared-memory map");
static_assert(KernelShape<false, false>::kSmemBytes <= 232448 && KernelShape<true, true>::kSmemBytes <= 232448,
              "shared memory budget");
static_assert(KernelShape<false, false>::kOffBar - KernelShape<false, false>::kOffOwn >= 4 * kQBoxBytes &&
                  KernelShape<true, false>::kOffBar - KernelShape<true, false>::kOffOwn >= 4 * kQBoxBytes,
              "the epilogue stages a 128 x 256 bf16 tile over the idle KV buffers");

struct VerifyParams {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* kv_bounds;
  const __nv_bfloat16* gate;
  __nv_bfloat16* out;
  float* lse;
  __nv_bfloat16* part_o;  // split partials o/l, bf16 [slot][rows][512]
  float* part_lse;
  int32_t* status;
  long long rows_total;  // T * H
  int R, q_per_req, H, max_pages, num_pages, num_splits, n_mtiles;
  float scale_log2;  // softmax_scale * log2(e)
  // balanced plan (units != nullptr): unit list and header written by the
  // plan kernel, the prerequisite grid of this launch
  const int4* units;
  const int* plan_header;
  long long part_w_stride;  // part_lse elements between consecutive slots
  int gate_dim;             // 512: elementwise gate [T][H][512]; 1: head-wise gate [T][H]
  float kv_scale;           // fp8 KV: the pool's scale (1 for bf16 KV)
  const uint8_t* kv8;       // fp8 KV: the e4m3 page pool [pages][64][512]
  long long part_lse_entries;  // part_lse elements the workspace holds (0 with one split)
  uint64_t wait_ns;             // short-wait instances: limit of every bounded wait (tests)
  // wave split mode (wave_s > 0): requests 0..wave_k-1 whole, the others in
  // wave_s uniform pieces whose partials go to slot (r - wave_k) wave_s + j
  int wave_k, wave_s;
};

// Two e4m3 codes (low byte first) -> two f16 (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_codes));
  return h2;
}

__device__ __forceinline__ int load_bound(const VerifyParams& p, int tok) {
  if (!SV_DCHECK(tok >= 0 && tok < p.R * p.q_per_req, p.status)) return 0;
  int b = __ldg(p.kv_bounds + tok);
  const int cap = p.max_pages * kTileN;
  if (b < 0 || b > cap) {
    if (p.status) atomicOr(p.status, SV_DEV_BAD_BOUND);
    b = b < 0 ? 0 : cap;
  }
  return b;
}

// Bounded wait taken by a whole warp; all lanes get the same answer.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status, uint64_t limit_ns) {
  const bool ok = mbar_wait<false>(bar, parity, abort_flag, status, limit_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Bounded wait used only while tearing down (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

// Context of an epilogue box group (see store_boxes).
struct EpilogueCtx {
  const VerifyParams* p;
  const CUtensorMap* tmap_out;
  const CUtensorMap* tmap_part;
  uint8_t* sptr;
  uint32_t sbase, tmem, gate_full;
  int off_own, off_q;
  volatile int* abort_flag;
  int warp, lane, half, m_tile, r, s_idx, slot, Mq;
  bool fused;
};

// Epilogue boxes [bx0, bx1) of this thread's TMEM row (row i of lane
// quadrant warp % 4): O times `scale` (= 1/l; < 0 when the unit produced no
// O, which stores zeros), gated when this unit finishes its rows (else the
// split partial), bf16, staged swizzled in the idle KV ring; after each box
// a named barrier over the 128 threads of the group and `leader` starts its
// TMA tensor store (rows past M are dropped).  Used by the long-unit
// instances, whose softmax warps and helper warps split the four boxes.
template <bool kStack, bool kShortWaits>
__device__ __forceinline__ void store_boxes(const EpilogueCtx& c, int bx0, int bx1, float scale, uint32_t bar_id,
                                            bool leader) {
  const int wq = c.warp & 3;
  const int i = wq * 32 + c.lane;
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const int f = c.m_tile * kMTile + (kStack ? (i & 63) : i);
  const bool valid = f < c.Mq;
  const long long row_g = (long long)c.r * c.Mq + f;
  const bool have_o = scale >= 0.f;
  const float inv_l = have_o ? scale : 0.f;
  uint8_t* const stage = c.sptr + c.off_own;
  const uint32_t row_off = (uint32_t)i * 128u;
  const uint32_t swz = (uint32_t)(i & 7);
  // gate: head-wise, one sigmoid per row; elementwise, the staged gate tile;
  // a partial is not gated (the merge gates)
  const bool row_gate = c.fused && c.p->gate_dim == 1;
  const bool elem_gate = c.fused && c.p->gate_dim != 1;
  float g_row = 1.f;
  if (row_gate) g_row = valid ? fast_sigmoid(__bfloat162float(c.p->gate[row_g])) : 0.f;
  const bool gate_ok = elem_gate && warp_wait(c.gate_full, 0, c.abort_flag, c.p->status,
                                                      kShortWaits ? c.p->wait_ns : kWaitTimeoutNs);
  const uint8_t* const gs = c.sptr + c.off_q;
  const uint32_t st0 = c.sbase + c.off_own;
#ifdef SPECVERIFY_DEBUG
  constexpr uint32_t kMapBytes = (uint32_t)KernelShape<false, false>::kSmemUsed;
  auto smem_in = [&](uint32_t a, uint32_t bytes) { return a >= c.sbase && a + bytes <= c.sbase + kMapBytes; };
#endif
  SV_DCHECK(bx0 >= 0 && bx1 <= 4 && (c.tmem & 0xFFFFu) + kTmemCols <= 512u && wq * 32 + 32 <= 128, c.p->status);
  SV_DCHECK(!row_gate || !valid || row_g < c.p->rows_total, c.p->status);
#pragma unroll 1
  for (int bx = bx0; bx < bx1; ++bx) {
    uint32_t va[32], vb[32];  // columns 64 bx .. +31 and 64 bx + 32 .. +63
    if (have_o) {
      tmem_ld32(c.tmem + lane_off + kTmemO + 64u * bx, va);
      tmem_ld32(c.tmem + lane_off + kTmemO + 64u * bx + 32u, vb);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) va[u] = vb[u] = 0u;
    }
    auto v = [&](int k) { return __uint_as_float(k < 32 ? va[k] : vb[k - 32]); };
    // 16-byte chunk u of the row holds columns 64 bx + 8u .. +7
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t off = (uint32_t)bx * kQBoxBytes + row_off + (((uint32_t)u ^ swz) << 4);
      uint32_t ow[4];
      if (elem_gate) {
        const bool g_in = SV_DCHECK(smem_in(c.sbase + c.off_q + off, 16), c.p->status);
        const uint4 graw = gate_ok && g_in ? *reinterpret_cast<const uint4*>(gs + off) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t gw[4] = {graw.x, graw.y, graw.z, graw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
          ow[e] = pack_bf16x2(v(8 * u + 2 * e) * inv_l * fast_sigmoid(gf.x),
                              v(8 * u + 2 * e + 1) * inv_l * fast_sigmoid(gf.y));
        }
      } else {
        const float fs = inv_l * g_row;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ow[e] = pack_bf16x2(v(8 * u + 2 * e) * fs, v(8 * u + 2 * e + 1) * fs);
      }
      if (SV_DCHECK(smem_in(st0 + off, 16), c.p->status))
        *reinterpret_cast<uint4*>(stage + off) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
    fence_proxy_async_smem();
    named_bar_sync(bar_id, 128);
    if (leader && SV_DCHECK(smem_in(st0 + bx * kQBoxBytes, kQBoxBytes), c.p->status)) {
      if constexpr (!kStack) {
        if (c.fused)
          tma_store_3d(c.tmap_out, st0 + bx * kQBoxBytes, c.half * kDHalf + bx * 64, c.m_tile * kMTile, c.r);
        else
          tma_store_4d(c.tmap_part, st0 + bx * kQBoxBytes, c.half * kDHalf + bx * 64, c.m_tile * kMTile,
                       (c.p->units || c.p->wave_s > 0) ? 0 : c.r, (c.p->units || c.p->wave_s > 0) ? c.slot : c.s_idx);
      } else {
        // staged rows 64h .. 64h+63 are latent 256h + 64bx .. +63 (64-row boxes)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t src = st0 + bx * kQBoxBytes + h * (kQBoxBytes / 2);
          if (c.fused)
            tma_store_3d(c.tmap_out, src, h * kDHalf + bx * 64, 0, c.r);
          else
            tma_store_4d(c.tmap_part, src, h * kDHalf + bx * 64, 0, (c.p->units || c.p->wave_s > 0) ? 0 : c.r,
                         (c.p->units || c.p->wave_s > 0) ? c.slot : c.s_idx);
        }
      }
      tma_store_commit();
    }
  }
}

// Tensor maps: tmap_kv 2-D over the page pool [pages*64][512] bf16; tmap_q,
// tmap_gate, tmap_out 3-D [R][M][512] bf16 (rows past a request's M fall out
// of bounds: zero on load, dropped on store); tmap_part 4-D [S][R][M][512] fp32.
// kShortWaits: the test instances, whose bounded waits give up after
// p.wait_ns instead of kWaitTimeoutNs (a compile-time limit costs the
// production instances nothing in their wait loops; a limit read from the
// parameters cost the long-context batch 2%).
template <bool kF8, bool kTwo, bool kStack, bool kShortWaits>
__global__ void __launch_bounds__(KernelShape<kF8, kTwo>::kThreads, 1)
    mla_verify_kernel(const __grid_constant__ CUtensorMap tmap_kv,
                      const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_gate,
                      const __grid_constant__ CUtensorMap tmap_out,
                      const __grid_constant__ CUtensorMap tmap_part, const VerifyParams p) {
  using K = KernelShape<kF8, kTwo>;
  const uint64_t wait_ns = kShortWaits ? p.wait_ns : kWaitTimeoutNs;
  constexpr int kOwnStages = K::kOwnStages, kOthStages = K::kOthStages, kNumBars = K::kNumBars;
  constexpr int kOffQ = K::kOffQ, kOffOwn = K::kOffOwn, kOffOth = K::kOffOth, kOffBar = K::kOffBar;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* const sptr = smem_raw + (sbase - raw);
  const uint32_t q_s = sbase + kOffQ;
  const uint32_t own0 = sbase + kOffOwn;
  const uint32_t oth0 = sbase + kOffOth;
  const uint32_t bar0 = sbase + kOffBar;
  auto own_full = [&](int s) { return bar0 + 8u * s; };
  auto own_empty = [&](int s) { return bar0 + 8u * (3 + s); };
  auto oth_full = [&](int s) { return bar0 + 8u * (6 + s); };
  auto oth_empty = [&](int s) { return bar0 + 8u * (8 + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (10 + b); };
  auto p_full = [&](int b) { return bar0 + 8u * (12 + b); };
  auto pv_done = [&](int b) { return bar0 + 8u * (14 + b); };
  const uint32_t q_ready = bar0 + 8u * 16;  // Q own half in TMEM + Q other half in SMEM
  const uint32_t drain_bar = bar0 + 8u * 17;
  const uint32_t drain_pv = bar0 + 8u * 22;  // the P V issuer's MMAs have completed
  const uint32_t drain_odd = bar0 + 8u * 23;  // the odd-tile score issuer's MMAs have completed
  const uint32_t gate_full = bar0 + 8u * 18;  // gate tile staged in the Q region
  const uint32_t q_tma = bar0 + 8u * 19;      // fp8 KV: bf16 query half landed (converted in place)
  // this CTA's query half, TMA-staged in the idle other-half ring, landed /
  // copied into TMEM (the ring slots may take KV tiles)
  const uint32_t q_own_full = bar0 + 8u * 20;
  const uint32_t q_own_free = bar0 + 8u * 21;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sptr + kOffBar + 8 * kNumBars);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sptr + kOffBar + 8 * kNumBars + 4);
#ifdef SPECVERIFY_DEBUG
  // debug build: this CTA's shared-memory map is [sbase, sbase + kSmemUsed)
  auto smem_in = [&](uint32_t a, uint32_t bytes) {
    return a >= sbase && a + bytes <= sbase + (uint32_t)K::kSmemUsed;
  };
  SV_DCHECK(sbase + (uint32_t)K::kSmemUsed <= raw + (uint32_t)K::kSmemBytes, p.status);
#endif

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // ---- the work unit: (request r, 128-row tile, latent half, KV tile range)
  int half, m_tile, r, s_idx = 0, plan_lo = 0, plan_hi = 0, slot = -1;
  bool fused;  // one piece: normalise + gate here, else write a partial
  const int S = p.num_splits;
  if (p.units) {
    // balanced plan: wait for the plan kernel, then read this CTA's unit
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if ((int)blockIdx.x >= ld_dep_s32(p.plan_header + 1)) return;  // spare CTA
    SV_DCHECK((long long)blockIdx.x < (long long)gridDim.x, p.status);
    const int4 u = ld_dep_i4(p.units + blockIdx.x);
    r = u.x;
    m_tile = u.y >> 1;
    half = u.y & 1;
    plan_lo = u.z & 0xFFFF;
    plan_hi = (int)((unsigned)u.z >> 16);
    slot = u.w;
    fused = slot < 0;
  } else if (p.wave_s > 0) {
    // wave split mode: the whole requests' units first (they fill the first
    // wave of CTAs), then the pieces of the others
    half = (int)(blockIdx.x & 1);
    const int unit = (int)(blockIdx.x >> 1);
    const int whole = p.wave_k * p.n_mtiles;
    if (unit < whole) {
      r = unit / p.n_mtiles;
      m_tile = unit % p.n_mtiles;
      fused = true;
    } else {
      const int q = unit - whole;
      const int rj = q / p.n_mtiles;
      m_tile = q % p.n_mtiles;
      r = p.wave_k + rj / p.wave_s;
      s_idx = rj % p.wave_s;
      slot = rj;
      fused = false;
    }
  } else {
    // latent half of O owned by this CTA (stacked: both, in the two lane halves)
    half = kStack ? 0 : (int)(blockIdx.x & 1);
    const int unit = kStack ? (int)blockIdx.x : (int)(blockIdx.x >> 1);
    s_idx = unit % S;
    const int rm = unit / S;
    m_tile = rm % p.n_mtiles;
    r = rm / p.n_mtiles;
    fused = (S == 1);
  }
  // partials addressed by slot ([slot][Mq] rows: balanced plan, wave mode) or
  // by (split, request) ([S][R][Mq] rows: uniform splits)
  const bool slotted = p.units != nullptr || p.wave_s > 0;
  const int Mq = p.H * p.q_per_req;
  SV_DCHECK(r >= 0 && r < p.R && m_tile >= 0 && m_tile < p.n_mtiles && (half == 0 || half == 1), p.status);
  SV_DCHECK(!p.units || (plan_lo <= plan_hi && plan_hi <= p.max_pages), p.status);
  SV_DCHECK(fused || (long long)(slotted ? slot : s_idx) * p.part_w_stride + (long long)(slotted ? 0 : r) * Mq +
                             Mq <= p.part_lse_entries, p.status);

  // warp 0: start the dependent loads of the set-up (bounds -> block table ->
  // KV tiles) from L2 rather than HBM: prefetch the request's bound and
  // block-table lines now
  if (warp == 0) {
    const int32_t* bt_row = p.block_table + (long long)r * p.max_pages;
    for (int j = lane * 32; j < p.max_pages; j += 32 * 32) prefetch_l2(bt_row + j);
    if (lane == 0) prefetch_l2(p.kv_bounds + r * p.q_per_req);
    if (lane == 1) prefetch_l2(p.kv_bounds + r * p.q_per_req + p.q_per_req - 1);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kOwnStages; ++s) {
      mbar_init(own_full(s), K::kFullCount);
      mbar_init(own_empty(s), 1);
    }
    for (int s = 0; s < kOthStages; ++s) {
      mbar_init(oth_full(s), K::kFullCount);
      mbar_init(oth_empty(s), 1);
    }

    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), 128);
      mbar_init(pv_done(b), 1);
    }
    // 128 softmax threads (the TMEM half), + the 128 converter threads with
    // fp8 KV (the other half, converted to f16); the bf16 other half is
    // waited for on q_tma
    mbar_init(q_ready, kF8 ? 128 + 128 : 128);
    mbar_init(drain_bar, 1);
    mbar_init(drain_pv, 1);
    mbar_init(drain_odd, 1);
    mbar_init(gate_full, 1);
    mbar_init(q_tma, 1);
    mbar_init(q_own_full, 1);
    mbar_init(q_own_free, 128);
    *abort_flag = 0;
    fence_mbar_init_cluster();
    // both latent halves of the unit's 128 query rows, at once (they depend
    // on the unit only): this CTA's half staged in the idle other-half ring
    // for the softmax warps to move into TMEM, the other half into its own
    // region (A of the SMEM score GEMM; fp8 KV: converted to f16 in place)
    if constexpr (!kStack) {
      mbar_arrive_expect_tx(q_own_full, kQHalfBytes);
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (SV_DCHECK(smem_in(oth0 + b * kQBoxBytes, kQBoxBytes), p.status))
          tma_load_3d(oth0 + b * kQBoxBytes, &tmap_q, q_own_full, half * kDHalf + b * 64, m_tile * kMTile, r);
      mbar_arrive_expect_tx(q_tma, kQHalfBytes);
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (SV_DCHECK(smem_in(q_s + b * kQBoxBytes, kQBoxBytes), p.status))
          tma_load_3d(q_s + b * kQBoxBytes, &tmap_q, q_tma, (1 - half) * kDHalf + b * 64, m_tile * kMTile, r);
    } else {
      // stacked: tmap_q has 64-row boxes.  Latent 0..255 of the (at most 64)
      // query rows into rows 0..63 of the staging boxes; latent 256..511
      // twice, into rows 0..63 and 64..127 of the SMEM A operand, so that
      // score rows L and L + 64 are the same query row.
      mbar_arrive_expect_tx(q_own_full, kQHalfBytes / 2);
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (SV_DCHECK(smem_in(oth0 + b * kQBoxBytes, kQBoxBytes / 2), p.status))
          tma_load_3d(oth0 + b * kQBoxBytes, &tmap_q, q_own_full, b * 64, 0, r);
      mbar_arrive_expect_tx(q_tma, kQHalfBytes);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (!SV_DCHECK(smem_in(q_s + b * kQBoxBytes, kQBoxBytes), p.status)) continue;
        tma_load_3d(q_s + b * kQBoxBytes, &tmap_q, q_tma, kDHalf + b * 64, 0, r);
        tma_load_3d(q_s + b * kQBoxBytes + kQBoxBytes / 2, &tmap_q, q_tma, kDHalf + b * 64, 0, r);
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
#ifdef SPECVERIFY_DEBUG
  // debug build: TMEM address a (lane << 16 | column) with `cols` columns
  // from it, and the 32 lanes from its lane, inside this CTA's allocation
  auto tmem_in = [&](uint32_t a, uint32_t cols) {
    const uint32_t c0 = tmem & 0xFFFFu, c = a & 0xFFFFu, ln = a >> 16;
    return c >= c0 && c + cols <= c0 + kTmemCols && ln + 32 <= 128 && (ln & 31) == 0;
  };
#endif

  // ---- unit geometry (every thread derives the same values)
  const int t_first = (m_tile * kMTile) / p.H;
  const int t_last = min((m_tile * kMTile + kMTile - 1) / p.H, p.q_per_req - 1);
  // one pass over the request's bounds, with the out-of-range report after
  // it (no side effect between the loads, so they overlap)
  int maxb_tile = 0, maxb_req = 0;
  {
    const int cap = p.max_pages * kTileN;
    bool bad = false;
    SV_DCHECK((long long)(r + 1) * p.q_per_req <= (long long)p.R * p.q_per_req, p.status);
    for (int t = 0; t < p.q_per_req; ++t) {
      const int b = __ldg(p.kv_bounds + r * p.q_per_req + t);
      bad |= (b < 0) | (b > cap);
      const int bc = min(max(b, 0), cap);
      maxb_req = max(maxb_req, bc);
      if (t >= t_first && t <= t_last) maxb_tile = max(maxb_tile, bc);
    }
    if (bad && p.status) atomicOr(p.status, SV_DEV_BAD_BOUND);
  }
  int lo = plan_lo, hi = plan_hi;
  if (!p.units) {
    const int n_r = (maxb_req + kTileN - 1) / kTileN;
    const int s_r = p.wave_s > 0 ? (fused ? 1 : p.wave_s) : S;  // this request's pieces
    lo = (int)((long long)s_idx * n_r / s_r);
    hi = (int)((long long)(s_idx + 1) * n_r / s_r);
  }
  const int hi_eff = min(hi, (maxb_tile + kTileN - 1) / kTileN);
  const int ntiles = max(0, hi_eff - lo);


  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      if constexpr (!kF8) {
      tma_prefetch_desc(&tmap_kv);
      int last_own[kOwnStages];
      int last_oth[kOthStages];
      for (int s = 0; s < kOwnStages; ++s) last_own[s] = -1;
      for (int s = 0; s < kOthStages; ++s) last_oth[s] = -1;
      for (int it = 0; it < ntiles; ++it) {
        const int j = lo + it;
        if (!SV_DCHECK(j >= 0 && j < p.max_pages, p.status)) break;
        int page = __ldg(p.block_table + (long long)r * p.max_pages + j);
        if (page < 0 || page >= p.num_pages) {
          if (p.status) atomicOr(p.status, SV_DEV_BAD_PAGE);
          page = 0;
        }
        // own half: scores and P V
        const int so = it % kOwnStages;
        const int ro = it / kOwnStages;
        if (ro > 0 && !mbar_wait<false>(own_empty(so), (ro - 1) & 1, abort_flag, p.status, wait_ns)) break;
        mbar_arrive_expect_tx(own_full(so), kHalfTileBytes);
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (SV_DCHECK(smem_in(own0 + so * kHalfTileBytes + b * kBoxBytes, kBoxBytes) && page < p.num_pages,
                        p.status))
            tma_load_2d(own0 + so * kHalfTileBytes + b * kBoxBytes, &tmap_kv, own_full(so),
                        half * kDHalf + b * 64, page * kTileN);
        last_own[so] = ro;
        // other half: scores only (its ring holds the staged query half until
        // the softmax warps have moved it into TMEM)
        const int sx = it % kOthStages;
        const int rx = it / kOthStages;
        if (it == 0 && !mbar_wait<false>(q_own_free, 0, abort_flag, p.status, wait_ns)) break;
        if (rx > 0 && !mbar_wait<false>(oth_empty(sx), (rx - 1) & 1, abort_flag, p.status, wait_ns)) break;
        mbar_arrive_expect_tx(oth_full(sx), kHalfTileBytes);
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (SV_DCHECK(smem_in(oth0 + sx * kHalfTileBytes + b * kBoxBytes, kBoxBytes) && page < p.num_pages,
                        p.status))
            tma_load_2d(oth0 + sx * kHalfTileBytes + b * kBoxBytes, &tmap_kv, oth_full(sx),
                        (1 - half) * kDHalf + b * 64, page * kTileN);
        last_oth[sx] = rx;
      }
      // every copy this CTA started has landed before teardown
      drain_wait(q_own_full, 0);
      drain_wait(q_tma, 0);
      for (int s = 0; s < kOwnStages; ++s)
        if (last_own[s] >= 0) drain_wait(own_full(s), last_own[s] & 1);
      for (int s = 0; s < kOthStages; ++s)
        if (last_oth[s] >= 0) drain_wait(oth_full(s), last_oth[s] & 1);
      } else {
        // fp8 KV: the converter warps fill the KV rings; the query copies have
        // to land before teardown
        drain_wait(q_own_full, 0);
        drain_wait(q_tma, 0);
      }
    } else if (lane == 0) {
      // an empty unit: only the query copies were started
      drain_wait(q_own_full, 0);
      drain_wait(q_tma, 0);
    }
    __syncwarp();
  } else if (warp == 1 || (kTwo && warp == K::kOddWarp)) {
    // ------------------------------------------------------------ score MMA issuers
    // Two warps: warp 1 the even tiles (score buffer 0), the other warp the
    // odd tiles (buffer 1).  Each buffer is written by one warp only, and the
    // tensor pipe takes MMAs from both (one issuing thread alone issues a
    // 128 x 64 x 16 MMA no faster than ~45 cycles; the datapath needs 32).
    // Short units keep one issuer (interleaving tiles 0 and 1 would delay the
    // first scores, which a short unit waits for).
    const bool two = kTwo && ntiles >= kTwoIssuerTiles;
    const int first = (warp == 1) ? 0 : 1;
    const int step = two ? 2 : 1;
    constexpr uint32_t idesc_s = kF8 ? idesc_f16_f32(128, 64, false, false) : idesc_bf16_f32(128, 64, false, false);
    const uint64_t q_desc = sdesc_sw128(q_s, 16, 1024);  // A of the other-half score MMAs
    bool ok = ntiles > 0 && (warp == 1 || two) && warp_wait(q_ready, 0, abort_flag, p.status, wait_ns) &&
              (kF8 || warp_wait(q_tma, 0, abort_flag, p.status, wait_ns));
    bool issued = false;
    auto zero_tail = [&](uint8_t* tile, int rows_valid) {
      // rows no query row of this unit may see: zero them (pool slack may be
      // NaN, and P V would turn 0 * NaN into NaN); lane = 4 rows x 8 chunks
      for (int rr = rows_valid + (lane >> 3); rr < kTileN; rr += 4) {
#pragma unroll
        for (int b = 0; b < 4; ++b)
          *reinterpret_cast<uint4*>(tile + b * kBoxBytes + rr * 128 + (lane & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    };
    if (ok) tc_fence_after();
    for (int it = first; ok && it < ntiles; it += step) {
      const int so = it % kOwnStages;
      const int sx = it % kOthStages;
      const int sb = it & 1;
      if (!warp_wait(own_full(so), (it / kOwnStages) & 1, abort_flag, p.status, wait_ns) ||
          !warp_wait(oth_full(sx), (it / kOthStages) & 1, abort_flag, p.status, wait_ns)) {
        ok = false;
        break;
      }
      // the score buffer is free once the P V of two tiles ago (which read
      // its P) has completed
      if (it >= 2 && !warp_wait(pv_done(sb), ((it - 2) >> 1) & 1, abort_flag, p.status, wait_ns)) {
        ok = false;
        break;
      }
      const int rows_valid = maxb_tile - (lo + it) * kTileN;
      SV_DCHECK(rows_valid > 0 && smem_in(own0 + so * kHalfTileBytes, kHalfTileBytes) &&
                    smem_in(oth0 + sx * kHalfTileBytes, kHalfTileBytes), p.status);
      if (rows_valid < kTileN) {
        // the own half is V of P V; the other half feeds only scores (its
        // slack columns are masked by selection), except in the stacked form
        zero_tail(sptr + kOffOwn + so * kHalfTileBytes, rows_valid);
        if constexpr (kStack) zero_tail(sptr + kOffOth + sx * kHalfTileBytes, rows_valid);
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint64_t ko_desc = sdesc_sw128(own0 + so * kHalfTileBytes, 16, 1024);
        const uint64_t kx_desc = sdesc_sw128(oth0 + sx * kHalfTileBytes, 16, 1024);
        const uint32_t ko_lo = (uint32_t)ko_desc, kx_lo = (uint32_t)kx_desc;
        const uint32_t k_hi = (uint32_t)(ko_desc >> 32);  // the same for every K-major operand
        const uint32_t q_lo = (uint32_t)q_desc;
        const uint32_t d = tmem + kTmemS + 64u * sb;
        const bool dbg_ok = SV_DCHECK(tmem_in(d, 64) && tmem_in(tmem + kTmemQ, 128) && smem_in(q_s, kQHalfBytes) &&
                                          smem_in(own0 + so * kHalfTileBytes, kHalfTileBytes) &&
                                          smem_in(oth0 + sx * kHalfTileBytes, kHalfTileBytes), p.status);
        // B = K tile, K-major, 128-byte swizzle: step 16 latent columns (32
        // bytes) inside a box, next box every 4 steps.
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          if (dbg_ok)
            mma_ts_w(d, tmem + kTmemQ + 8u * kk, ko_lo + (uint32_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4),
                     k_hi, idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          if (dbg_ok)
            mma_ss_w(d, q_lo + (uint32_t)(((kk >> 2) * kQBoxBytes + (kk & 3) * 32) >> 4), k_hi,
                     kx_lo + (uint32_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4), k_hi, idesc_s, 1u);
        }
        mma_commit(s_full(sb));
        if constexpr (!kStack) mma_commit(oth_empty(sx));  // stacked: P V reads it too
      }
      __syncwarp();
      issued = true;
    }
    if (issued && lane == 0) {
      const uint32_t drain = first == 0 ? drain_bar : drain_odd;
      mma_commit(drain);
      drain_wait(drain, 0);
    }
    __syncwarp();
  } else if (warp == K::kPvWarp) {
    // ------------------------------------------------------------ P V issuer
    // A second issuing warp: the tensor pipe takes MMAs from both, so the
    // P V products no longer wait in line behind the score MMAs' issue.
    // It is the only writer of O (accumulation order unchanged).
    constexpr uint32_t idesc_pv = kF8 ? idesc_f16_f32(128, 256, false, true) : idesc_bf16_f32(128, 256, false, true);
    bool issued = false;
    for (int i = 0; i < ntiles; ++i) {
      const int sb = i & 1;
      const int so = i % kOwnStages;
      const int sx = i % kOthStages;
      if (!warp_wait(p_full(sb), (i >> 1) & 1, abort_flag, p.status, wait_ns)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a = tmem + kTmemS + 64u * sb;
        const bool dbg_ok = SV_DCHECK(tmem_in(a, 64) && tmem_in(tmem + kTmemO, 256) &&
                                          smem_in(own0 + so * kHalfTileBytes, kHalfTileBytes) &&
                                          (!kStack || smem_in(oth0 + sx * kHalfTileBytes, kHalfTileBytes)),
                                      p.status);
        // descriptors differ only in the 14-bit start-address field, which
        // never carries (shared addresses < 256 KB): one add per MMA
        const uint64_t pv_desc0 = sdesc_sw128(own0 + so * kHalfTileBytes, kBoxBytes, 1024);
        const uint32_t pv_lo = (uint32_t)pv_desc0, pv_hi = (uint32_t)(pv_desc0 >> 32);
        if constexpr (kStack) {
          // P is block-diagonal over K = 128: lanes 64..127 hold [0 | P] and
          // accumulate latent 256..511 from the other ring's tile; lanes
          // 0..63 hold [P | 0] and accumulate latent 0..255 from the own
          // ring's tile below.  The other-ring steps go first so that their
          // slot (the shallower ring) is released as early as possible.
          const uint32_t px_lo = (uint32_t)sdesc_sw128(oth0 + sx * kHalfTileBytes, kBoxBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            if (dbg_ok)
              mma_ts_w(tmem + kTmemO, a + 32u + 8u * kk, px_lo + (uint32_t)((kk * 16 * 128) >> 4), pv_hi, idesc_pv,
                       (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(oth_empty(sx));
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // B = V tile (own half), MN-major: N = 256 latent columns in four
          // 64-wide boxes (LBO = box stride), K = 16 KV rows per step (SBO = 8-row stride).
          if (dbg_ok)
            mma_ts_w(tmem + kTmemO, a + 8u * kk, pv_lo + (uint32_t)((kk * 16 * 128) >> 4), pv_hi, idesc_pv,
                     (kStack || i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(own_empty(so));
        mma_commit(pv_done(sb));
      }
      __syncwarp();
      issued = true;
    }
    if (issued && lane == 0) {
      mma_commit(drain_pv);
      drain_wait(drain_pv, 0);
    }
    __syncwarp();
  } else if (!kF8 || warp < 6) {
    // ------------------------------------------------------------ softmax + epilogue
    const int wq = warp & 3;  // TMEM lane quadrant of this warp
    const int i = wq * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    // stacked: lane i holds query row i mod 64 and latent half i / 64 of O
    const int qi = kStack ? (i & 63) : i;
    const int f = m_tile * kMTile + qi;
    const bool valid = f < Mq;
    const int t_loc = valid ? f / p.H : 0;
    const long long row_g = (long long)r * Mq + f;
    const int b_i = valid ? load_bound(p, r * p.q_per_req + t_loc) : 0;

    if (ntiles > 0 && warp_wait(q_own_full, 0, abort_flag, p.status, wait_ns)) {
      // this CTA's half of the query row, staged by TMA (row i of box c at
      // c * 16 KB + 128 i, 16-byte chunks swizzled by i mod 8) -> TMEM (bf16
      // pairs per 32-bit column); rows past M arrived as zeros
      const uint8_t* const qrow = sptr + kOffOth + qi * 128;
      SV_DCHECK(smem_in(oth0 + qi * 128, 3 * kQBoxBytes + 128) && tmem_in(tmem + lane_off + kTmemQ, 128) &&
                    (lane_off >> 16) == (uint32_t)(wq * 32), p.status);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 w = *reinterpret_cast<const uint4*>(qrow + c * kQBoxBytes + (((uint32_t)u ^ (uint32_t)(i & 7)) << 4));
          v[4 * u + 0] = w.x;
          v[4 * u + 1] = w.y;
          v[4 * u + 2] = w.z;
          v[4 * u + 3] = w.w;
        }
        if constexpr (kF8) {
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = bf16x2_to_f16x2(v[u]);
        }
        tmem_st32(tmem + lane_off + kTmemQ + 32u * c, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
      mbar_arrive(q_own_free);  // the staging slots may take KV tiles
    }
    // Stage the gate tile (128 rows x 256 columns) into the Q region once no
    // score GEMM will read it again.
    bool gate_loaded = false;  // the leader started the gate tile's copy
    auto load_gate = [&]() {
      gate_loaded = true;
      mbar_arrive_expect_tx(gate_full, kQHalfBytes);
      if constexpr (!kStack) {
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (SV_DCHECK(smem_in(q_s + b * kQBoxBytes, kQBoxBytes), p.status))
            tma_load_3d(q_s + b * kQBoxBytes, &tmap_gate, gate_full, half * kDHalf + b * 64,
                        m_tile * kMTile, r);
      } else {
        // rows 64h .. 64h+63 of box b: latent 256h + 64b .. +63 (64-row boxes)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (!SV_DCHECK(smem_in(q_s + b * kQBoxBytes, kQBoxBytes), p.status)) continue;
          tma_load_3d(q_s + b * kQBoxBytes, &tmap_gate, gate_full, b * 64, 0, r);
          tma_load_3d(q_s + b * kQBoxBytes + kQBoxBytes / 2, &tmap_gate, gate_full, kDHalf + b * 64, 0, r);
        }
      }
    };
    // an empty unit stages the gate at once, after the query copy into the
    // same region has landed
    if (fused && p.gate_dim != 1 && ntiles == 0 && leader &&
        mbar_wait<false>(q_tma, 0, abort_flag, p.status, wait_ns))
      load_gate();

    float m_ref = -INFINITY;  // running max (log2 units) used for exponentiation
    float l_sum = 0.f;
    bool ok = true;
    for (int it = 0; it < ntiles; ++it) {
      const int sb = it & 1;
      const uint32_t par = (it >> 1) & 1;
      if (!warp_wait(s_full(sb), par, abort_flag, p.status, wait_ns)) { ok = false; break; }
      if (fused && p.gate_dim != 1 && it == ntiles - 1 && leader)
        load_gate();  // last score GEMM is done
      SV_DCHECK(tmem_in(tmem + lane_off + kTmemS + 64u * sb, 64) && tmem_in(tmem + lane_off + kTmemO, 256),
                p.status);
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
      const int lim = b_i - (lo + it) * kTileN;  // columns >= lim are masked
      if (__any_sync(0xFFFFFFFFu, lim < kTileN)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = (c < lim) ? x[c] : -INFINITY;
      }
      // row max of the raw scores in eight independent chains (a single
      // fmaxf chain over 64 columns is a long serial dependency); the scale
      // is positive, so the scaled maximum is the maximum times the scale
      float mx[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mx[c] = fmaxf(x[c], x[c + 8]);
#pragma unroll
      for (int c = 16; c < 64; ++c) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) mx[c] = fmaxf(mx[c], mx[c + 4]);
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
      // lazy rescale: move the reference max only when it grows by > 2^8
      const bool move = tmax > m_ref + kRescaleThreshold;
      const float m_new = move ? tmax : m_ref;
      const bool rescale_o = move && (m_ref != -INFINITY);
      const float alpha = rescale_o ? exp2f(m_ref - m_new) : 1.0f;
      if (__any_sync(0xFFFFFFFFu, rescale_o)) {
        // O holds tiles < it: wait for PV(it-1), then scale the row in TMEM
        if (!warp_wait(pv_done((it - 1) & 1), ((it - 1) >> 1) & 1, abort_flag, p.status, wait_ns)) {
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
      // p = 2^(scale x - m) with one fma feeding the exp2 (a masked x is
      // -inf and gives 0); the row sum in eight independent chains
      float ps[8];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = fast_exp2(fmaf(x[2 * c], p.scale_log2, -msub));
        const float p1 = fast_exp2(fmaf(x[2 * c + 1], p.scale_log2, -msub));
        ps[c & 7] = (c < 8) ? p0 + p1 : ps[c & 7] + (p0 + p1);
        pk[c] = kF8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
      }
      l_sum += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      if constexpr (!kStack) {
        tmem_st32(tmem + lane_off + kTmemS + 64u * sb, pk);  // P over the consumed scores
      } else {
        // block-diagonal A of the stacked P V: [P | 0] in lanes 0..63, [0 | P]
        // in lanes 64..127 (K = 128: this tile's 64 KV rows twice)
        uint32_t zero[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) zero[c] = 0u;
        const uint32_t pcol = (i < 64) ? 0u : 32u;
        tmem_st32(tmem + lane_off + kTmemS + 64u * sb + pcol, pk);
        tmem_st32(tmem + lane_off + kTmemS + 64u * sb + (32u - pcol), zero);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full(sb));
    }

    // ---- epilogue: O/l as bf16 (gated when this unit finishes its rows, else
    // the split partial), one 64-column box at a time (store_boxes); with
    // helper warps the softmax warps do boxes 0..1 and hand 1/l over
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // a dependent merge may launch
    if (ok && ntiles > 0)
      ok = warp_wait(pv_done((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1, abort_flag, p.status, wait_ns);
    tc_fence_after();
    const bool have_o = ok && ntiles > 0;
    float inv_l = (l_sum > 0.f) ? 1.0f / l_sum : 0.f;
    if constexpr (kF8) inv_l *= p.kv_scale;  // o of the codes -> o of the rows
    const float lse_v = (l_sum > 0.f) ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
    if constexpr (K::kHelp) {
      const float scale = have_o ? inv_l : -1.f;
      // boxes 2..3 of the row go to the helper warp of this lane quadrant
      reinterpret_cast<float*>(sptr + K::kOffRowScale)[i] = scale;
      tc_fence_before();
      named_bar_sync(kHandoffBarId, 256);
      const EpilogueCtx ctx{&p, &tmap_out, &tmap_part, sptr, sbase, tmem, gate_full, kOffOwn, kOffQ, abort_flag,
                            warp, lane, half, m_tile, r, s_idx, slot, Mq, fused};
      store_boxes<kStack, kShortWaits>(ctx, 0, 2, scale, kEpilogueBarId, leader);
    } else {
    // the same box loop as store_boxes, all four boxes
    // staging: the KV rings are idle once the last P V has completed
    uint8_t* const stage = sptr + kOffOwn;
    const uint32_t row_off = (uint32_t)i * 128u;
    const uint32_t swz = (uint32_t)(i & 7);
    // gate: head-wise, one sigmoid per row; elementwise, the staged gate tile;
    // a partial is not gated (the merge gates)
    const bool row_gate = fused && p.gate_dim == 1;
    const bool elem_gate = fused && p.gate_dim != 1;
    float g_row = 1.f;
    SV_DCHECK(!row_gate || !valid || row_g < p.rows_total, p.status);
    if (row_gate) g_row = valid ? fast_sigmoid(__bfloat162float(p.gate[row_g])) : 0.f;
    const bool gate_ok = elem_gate && warp_wait(gate_full, 0, abort_flag, p.status, wait_ns);
    const uint8_t* const gs = sptr + kOffQ;
    const uint32_t st0 = sbase + kOffOwn;
    SV_DCHECK(tmem_in(tmem + lane_off + kTmemO, 256), p.status);
#pragma unroll 1
    for (int bx = 0; bx < 4; ++bx) {
      uint32_t va[32], vb[32];  // columns 64 bx .. +31 and 64 bx + 32 .. +63
      if (have_o) {
        tmem_ld32(tmem + lane_off + kTmemO + 64u * bx, va);
        tmem_ld32(tmem + lane_off + kTmemO + 64u * bx + 32u, vb);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) va[u] = vb[u] = 0u;
      }
      auto v = [&](int c) { return __uint_as_float(c < 32 ? va[c] : vb[c - 32]); };
      // 16-byte chunk u of the row holds columns 64 bx + 8u .. +7
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t off = (uint32_t)bx * kQBoxBytes + row_off + (((uint32_t)u ^ swz) << 4);
        uint32_t ow[4];
        if (elem_gate) {
          const bool g_in = SV_DCHECK(smem_in(q_s + off, 16), p.status);
          const uint4 graw =
              gate_ok && g_in ? *reinterpret_cast<const uint4*>(gs + off) : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t gw[4] = {graw.x, graw.y, graw.z, graw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
            ow[e] = pack_bf16x2(v(8 * u + 2 * e) * inv_l * fast_sigmoid(gf.x),
                                v(8 * u + 2 * e + 1) * inv_l * fast_sigmoid(gf.y));
          }
        } else {
          const float f = inv_l * g_row;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ow[e] = pack_bf16x2(v(8 * u + 2 * e) * f, v(8 * u + 2 * e + 1) * f);
        }
        if (SV_DCHECK(smem_in(st0 + off, 16), p.status))
          *reinterpret_cast<uint4*>(stage + off) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(kEpilogueBarId, 128);
      if (leader && SV_DCHECK(smem_in(st0 + bx * kQBoxBytes, kQBoxBytes), p.status)) {
        if constexpr (!kStack) {
          if (fused)
            tma_store_3d(&tmap_out, st0 + bx * kQBoxBytes, half * kDHalf + bx * 64, m_tile * kMTile, r);
          else
            tma_store_4d(&tmap_part, st0 + bx * kQBoxBytes, half * kDHalf + bx * 64, m_tile * kMTile,
                         slotted ? 0 : r, slotted ? slot : s_idx);
        } else {
          // staged rows 64h .. 64h+63 are latent 256h + 64bx .. +63 (64-row boxes)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t src = st0 + bx * kQBoxBytes + h * (kQBoxBytes / 2);
            if (fused)
              tma_store_3d(&tmap_out, src, h * kDHalf + bx * 64, 0, r);
            else
              tma_store_4d(&tmap_part, src, h * kDHalf + bx * 64, 0, slotted ? 0 : r, slotted ? slot : s_idx);
          }
        }
        tma_store_commit();
      }
    }
    }
    if (valid && (kStack ? i < 64 : half == 0)) {
      if (fused) {
        if (SV_DCHECK(row_g >= 0 && row_g < p.rows_total, p.status)) p.lse[row_g] = lse_v;
      } else {
        const long long w = slotted ? slot : s_idx;
        const long long z = slotted ? 0 : r;
        const long long e = w * p.part_w_stride + z * Mq + f;
        if (SV_DCHECK(e >= 0 && e < p.part_lse_entries, p.status)) p.part_lse[e] = lse_v;
      }
    }
    if (leader) tma_store_wait_read();  // SMEM stays valid until the stores have read it
    // the gate tile's copy has landed before teardown, even when a wait gave
    // up and the epilogue did not use it
    if (leader && gate_loaded) drain_wait(gate_full, 0);
    __syncwarp();
  }

  if constexpr (kF8) {
    if (warp >= 6 && warp < 10) {
      // ---------------------------------------------------------- fp8 converters
      // 128 threads.  First the other latent half of the unit's query rows
      // (TMA-loaded as bf16) is converted to f16 in shared memory.  Then the
      // KV: tile it's 64 x 512 codes are loaded into
      // registers while tile it-1 is converted (thread ct holds 16 chunks of 16
      // codes: row 4k + ct/32, columns 16 (ct%32) .. +15), then written as f16
      // into the own / other ring slots of tile it, swizzled like a TMA box.
      const int ct = threadIdx.x - 192;
      const int32_t* bt_row = p.block_table + (long long)r * p.max_pages + lo;
      uint4 buf[16];
      auto load_tile = [&](int it) {
        SV_DCHECK(lo + it >= 0 && lo + it < p.max_pages, p.status);
        int page = __ldg(bt_row + it);
        if (page < 0 || page >= p.num_pages) {
          if (ct == 0 && p.status) atomicOr(p.status, SV_DEV_BAD_PAGE);
          page = 0;
        }
        const uint4* base = reinterpret_cast<const uint4*>(p.kv8 + (long long)page * kTileN * kD);
#pragma unroll
        for (int k = 0; k < 16; ++k) buf[k] = __ldcs(base + (k * 128 + ct));
      };
      bool ok = true;
      if (ntiles > 0) {
        load_tile(0);
        // the bf16 query half -> f16 in place (elementwise, so the swizzle
        // is kept); rows past M arrived as zeros
        ok = mbar_wait<false>(q_tma, 0, abort_flag, p.status, wait_ns);
        if (ok) {
          uint4* const qs = reinterpret_cast<uint4*>(sptr + kOffQ);
          SV_DCHECK(smem_in(q_s, kQHalfBytes), p.status);
#pragma unroll 4
          for (int u = 0; u < kQHalfBytes / 16 / 128; ++u) {
            const uint4 w = qs[u * 128 + ct];
            qs[u * 128 + ct] = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y),
                                          bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
          }
          fence_proxy_async_smem();  // the tensor cores read what the threads wrote
          mbar_arrive(q_ready);
        }
        // the other-half ring holds the staged query half until the softmax
        // warps have moved it into TMEM
        if (ok) ok = mbar_wait<false>(q_own_free, 0, abort_flag, p.status, wait_ns);
      }
      for (int it = 0; ok && it < ntiles; ++it) {
        const int so = it % kOwnStages, ro = it / kOwnStages;
        const int sx = it % kOthStages, rx = it / kOthStages;
        if (ro > 0) ok = mbar_wait<false>(own_empty(so), (ro - 1) & 1, abort_flag, p.status, wait_ns);
        if (ok && rx > 0) ok = mbar_wait<false>(oth_empty(sx), (rx - 1) & 1, abort_flag, p.status, wait_ns);
        if (!ok) break;
        uint8_t* const own_t = sptr + kOffOwn + so * kHalfTileBytes;
        uint8_t* const oth_t = sptr + kOffOth + sx * kHalfTileBytes;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int c = k * 128 + ct;
          const int row = c >> 5, g = c & 31;  // 16-column group g of row `row`
          const uint4 v = buf[k];
          const int col = g * 16;
          uint8_t* const ring = ((col >> 8) == half) ? own_t : oth_t;
          const int b = (col & 255) >> 6;
          const int j0 = (col & 63) >> 3;  // 16-byte chunks j0, j0+1 of the 128-byte row
          uint4 w0, w1;
          w0.x = e4m3x2_to_f16x2(v.x);
          w0.y = e4m3x2_to_f16x2(v.x >> 16);
          w0.z = e4m3x2_to_f16x2(v.y);
          w0.w = e4m3x2_to_f16x2(v.y >> 16);
          w1.x = e4m3x2_to_f16x2(v.z);
          w1.y = e4m3x2_to_f16x2(v.z >> 16);
          w1.z = e4m3x2_to_f16x2(v.w);
          w1.w = e4m3x2_to_f16x2(v.w >> 16);
          uint8_t* const rb = ring + b * kBoxBytes + row * 128;
          if (SV_DCHECK(smem_in(smem_u32(rb), 128) && row < kTileN, p.status)) {
            *reinterpret_cast<uint4*>(rb + (((uint32_t)j0 ^ (uint32_t)(row & 7)) << 4)) = w0;
            *reinterpret_cast<uint4*>(rb + (((uint32_t)(j0 + 1) ^ (uint32_t)(row & 7)) << 4)) = w1;
          }
        }
        fence_proxy_async_smem();  // the tensor cores read what the threads wrote
        mbar_arrive(own_full(so));
        mbar_arrive(oth_full(sx));
        if (it + 1 < ntiles) load_tile(it + 1);
      }
    }
  }

  if constexpr (K::kHelp) {
    if (K::is_helper(warp)) {
      // ---------------------------------------------------------- epilogue helpers
      // after the softmax warps have seen the last P V complete
      named_bar_sync(kHandoffBarId, 256);
      tc_fence_after();
      const bool hl = (warp == K::kHelperLeaderWarp && lane == 0);
      const EpilogueCtx ctx{&p, &tmap_out, &tmap_part, sptr, sbase, tmem, gate_full, kOffOwn, kOffQ, abort_flag,
                            warp, lane, half, m_tile, r, s_idx, slot, Mq, fused};
      store_boxes<kStack, kShortWaits>(ctx, 2, 4, reinterpret_cast<const float*>(sptr + K::kOffRowScale)[(warp & 3) * 32 + lane],
                          kHelperBarId, hl);
      if (hl) tma_store_wait_read();  // SMEM stays valid until the stores have read it
      __syncwarp();
    }
  }

  // ---- teardown (every warp is converged here)
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ balanced plan
// One CTA turns the per-token bounds into the unit list of the attention
// kernel.  Request r needs n_r = ceil(max_t b_t / 64) KV tiles; a piece of a
// request is `upp` units (two-CTA form: n_mt row tiles x two latent halves;
// stacked form: one CTA), so the whole batch is upp * sum_r n_r CTA-tiles of
// work.  Pieces of c tiles,
//   c = max(ceil(sum_r n_r * wm / (SMs * wd)), ceil(max_r n_r / SV_MAX_SPLITS)),
// with wm = n_mt, wd = 1 (two-CTA: about two units per SM) or wm = 1, wd =
// kStackPlanDiv (stacked: about one unit per SM, whose units are short and
// pay their fixed cost once); request r gets s_r = max(1, ceil(n_r / c))
// pieces (the last one shorter).  Units are listed longest first (a counting
// sort over piece lengths), so the block scheduler hands the long pieces out
// before the short ones.  A request with one piece is finished by its units
// (normalise + gate); the others write partials to slots plan_base[r] + j.
// Layout of the plan area: header {c, n_units, n_slots}, splits[R],
// base[R], units[units_max] (int4: r, m_tile << 1 | half (stacked: 0),
// lo | hi << 16, slot or -1).
constexpr int kPlanThreads = 1024;
constexpr int kLenBuckets = 1024;

__device__ __forceinline__ int plan_bound(const int32_t* kv_bounds, int tok, int cap) {
  const int b = __ldg(kv_bounds + tok);
  return b < 0 ? 0 : (b > cap ? cap : b);
}

template <typename T>
__device__ T block_reduce(T v, T* s_red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const T x = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = is_max ? (x > v ? x : v) : v + x;
  }
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < nw ? s_red[lane] : (T)0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const T x = __shfl_xor_sync(0xFFFFFFFFu, v, o);
      v = is_max ? (x > v ? x : v) : v + x;
    }
    if (lane == 0) s_red[0] = v;
  }
  __syncthreads();
  const T r = s_red[0];
  __syncthreads();
  return r;
}

// Exclusive prefix sum over the block (one value per thread, thread order).
__device__ int block_excl_scan(int v, int* s_scan, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? s_scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) s_scan[32 + lane] = w;
  }
  __syncthreads();
  const int res = (warp > 0 ? s_scan[32 + warp - 1] : 0) + incl - v;
  *total = s_scan[32 + nw - 1];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t* __restrict__ kv_bounds, int R, int q_per_req, int max_pages,
                int upp, int wm, int wd, int sms, int units_max, int slots_max, int* __restrict__ header,
                int* __restrict__ splits, int* __restrict__ base, int4* __restrict__ units,
                int32_t* __restrict__ status) {
  __shared__ long long s_red64[32];
  __shared__ int s_red[32];
  __shared__ int s_scan[64];
  __shared__ int s_cnt[kLenBuckets];
  // the attention CTAs may take their SMs now; they wait for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  const int cap = max_pages * kTileN;
  // 1. KV tiles per request (kept in `splits` until step 4)
  long long psum = 0;
  int pmax = 0;
  for (int r = tid; r < R; r += kPlanThreads) {
    int mb = 0;
    for (int t = 0; t < q_per_req; ++t) mb = max(mb, plan_bound(kv_bounds, r * q_per_req + t, cap));
    const int n = (mb + kTileN - 1) / kTileN;
    splits[r] = n;
    psum += n;
    pmax = max(pmax, n);
  }
  psum = block_reduce<long long>(psum, s_red64, false);
  pmax = block_reduce<int>(pmax, s_red, true);
  long long c = (psum * wm + (long long)sms * wd - 1) / ((long long)sms * wd);
  c = max(c, (long long)(pmax + SV_MAX_SPLITS - 1) / SV_MAX_SPLITS);
  if (c < 1) c = 1;
  // 2. pieces per request, slots, and piece-length histogram
  for (int b = tid; b < kLenBuckets; b += kPlanThreads) s_cnt[b] = 0;
  __syncthreads();
  int carry_slots = 0, carry_units = 0;
  for (int r0 = 0; r0 < R; r0 += kPlanThreads) {
    const int r = r0 + tid;
    int n = 0, sr = 0;
    if (r < R) {
      n = splits[r];
      sr = n == 0 ? 1 : (int)((n + c - 1) / c);
      for (int j = 0; j < sr; ++j) {
        const int len = (j < sr - 1) ? (int)c : n - (int)((sr - 1) * c);
        const int bk = (int)((long long)len * (kLenBuckets - 1) / c);
        atomicAdd(&s_cnt[bk], upp);
      }
    }
    int tot = 0;
    const int b_excl = block_excl_scan(sr >= 2 ? sr : 0, s_scan, &tot);
    if (r < R) base[r] = carry_slots + b_excl;
    carry_slots += tot;
    int tu = 0;
    block_excl_scan(sr, s_scan, &tu);
    carry_units += tu * upp;
  }
  __syncthreads();
  // 3. start of every length bucket, longest first (bucket kLenBuckets-1 first)
  {
    const int b = kLenBuckets - 1 - tid;  // thread tid owns the tid-th longest bucket
    const int v = (tid < kLenBuckets) ? s_cnt[b] : 0;
    int tot = 0;
    const int st = block_excl_scan(v, s_scan, &tot);
    if (tid < kLenBuckets) s_cnt[b] = st;
  }
  __syncthreads();
  const bool fits = carry_units <= units_max && carry_slots <= slots_max;
  if (!fits && tid == 0 && status) atomicOr(status, SV_DEV_BAD_BOUND);
  // 4. place the units
  for (int r = tid; fits && r < R; r += kPlanThreads) {
    const int n = splits[r];
    const int sr = n == 0 ? 1 : (int)((n + c - 1) / c);
    for (int j = 0; j < sr; ++j) {
      const int plo = (int)(j * c);
      const int phi = (j < sr - 1) ? (int)((j + 1) * c) : n;
      const int bk = (int)((long long)(phi - plo) * (kLenBuckets - 1) / c);
      const int pos = atomicAdd(&s_cnt[bk], upp);
      const int sl = sr >= 2 ? base[r] + j : -1;
      for (int u = 0; u < upp; ++u)
        if (SV_DCHECK(pos + u >= 0 && pos + u < units_max && sl < slots_max, status))
          units[pos + u] = make_int4(r, u, plo | (phi << 16), sl);
    }
  }
  __syncthreads();
  // a plan that does not fit the plan area (reported above) places no unit
  // and leaves every request at one piece, so the merge reads no slot
  for (int r = tid; r < R; r += kPlanThreads) {
    const int n = splits[r];
    splits[r] = (n == 0 || !fits) ? 1 : (int)((n + c - 1) / c);
  }
  if (tid == 0) {
    header[0] = (int)c;
    header[1] = fits ? carry_units : 0;
    header[2] = carry_slots;
  }
}

// ------------------------------------------------------------------ host side
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
bool g_attr_set[kMaxDevices];
std::mutex g_dev_mu;

// Every instance of the attention kernel: index kv_fp8 | two << 1 |
// stack << 2 | short_waits << 3.
using VerifyKernel = decltype(&mla_verify_kernel<false, false, false, false>);
template <size_t... I>
constexpr std::array<VerifyKernel, sizeof...(I)> verify_kernels(std::index_sequence<I...>) {
  return {&mla_verify_kernel<(I & 1) != 0, (I & 2) != 0, (I & 4) != 0, (I & 8) != 0>...};
}
constexpr auto kVerifyKernels = verify_kernels(std::make_index_sequence<16>{});

bool device_setup(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_attr_set[dev]) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    constexpr int smem = KernelShape<false, false>::kSmemBytes;  // the same for every instance
    constexpr auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    for (const VerifyKernel k : kVerifyKernels)
      if (cudaFuncSetAttribute(k, attr, smem) != cudaSuccess) return false;
    g_sm_count[dev] = sms;
    g_attr_set[dev] = true;
  }
  if (sm_count) *sm_count = g_sm_count[dev];
  return true;
}

// The stacked instance (both latent halves in one CTA, stacked in the TMEM
// lanes) serves requests of at most 64 query rows.  Its KV rings are two
// tiles deep (a tile holds both ring slots until its P V completes), so it
// pays only when a unit holds several tiles: measured on the C = 64 plain
// decode batch (20 tiles per request) 47.5 us against 51.0 us for the
// two-CTA form, and slower than it on 1-2 tile units.  The caller picks the
// form per call (SV_FORM_*); the automatic choice takes the stacked form for
// units of at least kStackMinTiles tiles.
constexpr int kStackMinTiles = 4;
inline bool valid_form(int form) {
  return form == SV_FORM_AUTO || form == SV_FORM_TWO_CTA || form == SV_FORM_STACKED;
}
// Stacked form for units of ceil(max_pages / S) tiles?
inline bool use_stack(long long Mq, long long max_pages, long long S, int form) {
  if (Mq > 64 || form == SV_FORM_TWO_CTA) return false;
  return form == SV_FORM_STACKED || (max_pages + S - 1) / S >= kStackMinTiles;
}
// The same under the balanced plan, whose pieces hold ceil(sum n_r / SMs)
// tiles or more (the stacked form's units are one per SM).
inline bool use_stack_balanced(long long Mq, int form) { return Mq <= 64 && form != SV_FORM_TWO_CTA; }
// Stacked units per SM the balanced plan aims at (pieces of
// ceil(sum n_r / (SMs * kStackPlanDiv)) tiles).  plan_layout and
// plan_workspace_bound hold at most kStackPlanDiv * SMs + R + 1 pieces.
// Measured on 16 plain-decode requests of 8K-32K positions (GB300): one
// unit per SM 99-100 us, two 116 us, the two-CTA form's plan 122 us.
// (Raising c further until every unit fits one wave measured slower.)
constexpr int kStackPlanDiv = 1;
static_assert(kStackPlanDiv >= 1 && kStackPlanDiv <= 2, "the plan area is sized for at most two units per SM");

// Splits: enough (request, row tile, split, latent half) CTAs to fill the SMs
// once, each split keeping at least 2 KV tiles (on the C = 1 verify batch,
// 24 tiles: 12 splits 22.7 us, 8: 22.9, 6: 24.7, 19: 24.9 measured).  A
// stacked unit is one CTA per (request, split).
int fill_splits(long long ctas_per_split, int max_pages, int sm_count) {
  if (ctas_per_split <= 0) return 1;
  long long s = (long long)sm_count / ctas_per_split;
  const long long by_len = max_pages / 2;
  if (s > by_len) s = by_len;
  if (s > SV_MAX_SPLITS) s = SV_MAX_SPLITS;
  if (s < 1) s = 1;
  return (int)s;
}
int auto_splits(int R, int q_per_req, int H, int max_pages, int sm_count, int form) {
  const long long Mq = (long long)H * q_per_req;
  const long long n_mt = (Mq + kMTile - 1) / kMTile;
  // the stacked form if its own split count leaves it long enough units
  const int s_stack = fill_splits((long long)R * n_mt, max_pages, sm_count);
  if (use_stack(Mq, max_pages, s_stack, form)) return s_stack;
  return fill_splits(2ll * R * n_mt, max_pages, sm_count);
}

// Wave split mode, for batches whose unsplit units (2 per row tile) fill the
// SMs more than once but less than twice: the first k requests stay whole
// and fill the first wave, the other R - k are cut into s uniform pieces that
// fill the second wave, so no SM idles behind a second round of whole
// requests while every unit still pays its fixed cost only once or twice.
//   k = floor(SMs / (2 n_mt)),   s = max(2, floor(SMs / (2 n_mt (R - k)))),
// each piece keeping at least 2 KV tiles.  False when the mode does not
// apply (one wave or more than two, fewer than 4 tiles per request).
inline bool wave_params(long long R, long long n_mt, long long max_pages, int sms, int* k, int* s) {
  const long long units = 2 * n_mt * R;
  if (units <= sms || units >= 2ll * sms || max_pages < 4) return false;
  const long long kk = sms / (2 * n_mt);
  if (kk < 1 || kk >= R) return false;
  long long ss = sms / (2 * n_mt * (R - kk));
  if (ss < 2) ss = 2;
  if (ss > max_pages / 2) ss = max_pages / 2;
  if (ss > SV_MAX_SPLITS) ss = SV_MAX_SPLITS;
  if (ss < 2) return false;
  *k = (int)kk;
  *s = (int)ss;
  return true;
}

inline bool misaligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0;
}

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

int current_sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
    return v;
  return 152;
}

// Balanced-plan workspace: header, splits[R], base[R], units, then the
// partials of at most slots_max pieces ([slots][Mq][512] fp32 + [slots][Mq]).
struct PlanLayout {
  size_t splits, base, units, part_o, part_lse, total;
  int units_max, slots_max;
};
PlanLayout plan_layout(int R, int Mq, int n_mt, int sms, bool stack) {
  PlanLayout L;
  // two-CTA pieces: sum_r s_r <= sum n_r / c + R <= SMs / n_mt + R, 2 n_mt
  // units each; stacked pieces: <= kStackPlanDiv SMs + R, one unit each
  L.units_max = stack ? kStackPlanDiv * sms + R + 1 : 2 * sms + 2 * n_mt * R;
  L.slots_max = stack ? kStackPlanDiv * sms + R + 1 : sms / n_mt + R + 1;
  L.splits = 256;
  L.base = L.splits + align256((size_t)R * 4);
  L.units = L.base + align256((size_t)R * 4);
  L.part_o = L.units + align256((size_t)L.units_max * 16);
  L.part_lse = L.part_o + align256((size_t)L.slots_max * Mq * kD * 2);
  L.total = L.part_lse + align256((size_t)L.slots_max * Mq * 4);
  return L;
}
// An upper bound of plan_layout(...).total from T = R*q_per_req and H only
// (two-CTA: n_mt * R <= T*H/128 + R, slots * Mq <= 128*sms + 2*T*H; stacked,
// Mq <= 64: pieces <= 2*sms + R + 1 <= 2*sms + 2*T, slots * Mq <= 128*sms +
// 2*T*H).
size_t plan_workspace_bound(long long T, long long H, int sms) {
  const long long rows = T * H;
  const long long units_max = 2ll * sms + 2 * (rows / 128 + T);
  const long long slot_rows = 128ll * sms + 2 * rows;
  return 256 + 2 * align256((size_t)T * 4) + align256((size_t)units_max * 16) +
         align256((size_t)slot_rows * kD * 2) + align256((size_t)slot_rows * 4) + 1024;
}

}  // namespace
}  // namespace sv

// Automatic choice.  A unit costs about 8 KV tiles of fixed set-up and
// epilogue (measured on GB300: ~12 us against ~1.6 us per tile), so cutting
// requests into pieces pays only for long contexts: the balanced plan is used
// when the requests' row tiles fit the SMs once (so uniform splits would
// leave SMs idle behind the longest request) and a request may hold at least
// 64 tiles (4096 positions); otherwise uniform splits.
extern "C" int sv_mla_verify_num_splits(int R, int q_per_req, int H, int max_pages_per_req, int form) {
  if (!sv::valid_form(form)) return 0;
  const int sms = sv::current_sm_count();
  const long long n_mt = ((long long)H * q_per_req + sv::kMTile - 1) / sv::kMTile;
  if (R >= 2 && max_pages_per_req >= 64 && max_pages_per_req <= 0xFFFF && 2 * n_mt * R <= sms)
    return SV_SPLITS_BALANCED;
  // the wave mode for batches of two-CTA units between one and two waves
  // of the SMs (the C = 32 verify batch: 72.4 -> 62.1 us on GB300; other
  // (k, s) measured 62.1-66.2 us)
  int wk = 0, ws = 0;
  if (form != SV_FORM_STACKED && !(H * (long long)q_per_req <= 64 && form == SV_FORM_AUTO) &&
      sv::wave_params(R, n_mt, max_pages_per_req, sms, &wk, &ws))
    return SV_SPLITS_WAVE;
  return sv::auto_splits(R, q_per_req, H, max_pages_per_req, sms, form);
}

extern "C" size_t sv_mla_verify_workspace_bytes(int T, int H, int num_splits) {
  if (T <= 0 || H <= 0) return 0;
  if (num_splits == SV_SPLITS_BALANCED) return sv::plan_workspace_bound(T, H, sv::current_sm_count());
  if (num_splits == SV_SPLITS_WAVE) {
    // slots * Mq <= (R - k) s Mq <= max(SMs / (2 n_mt), 2 (R - k)) * 128 n_mt
    //            <= 64 SMs + 2 T H rows (Mq <= 128 n_mt, (R - k) Mq <= T H)
    const size_t slot_rows = (size_t)64 * sv::current_sm_count() + 2 * (size_t)T * (size_t)H;
    return sv::align256(slot_rows * sv::kD * sizeof(__nv_bfloat16)) + slot_rows * sizeof(float);
  }
  if (num_splits <= 1) return 0;
  const size_t rows = (size_t)T * (size_t)H;
  const size_t o_bytes = (size_t)num_splits * rows * sv::kD * sizeof(__nv_bfloat16);
  return o_bytes + (size_t)num_splits * rows * sizeof(float);
}

namespace sv {
namespace {
// The attention call for both KV formats: kv_fp8 selects an e4m3 page pool
// with scale kv_scale (the fp8 kernel variant), else a bf16 pool.
sv_status verify_impl(const void* q_latent, const void* kv_pages, bool kv_fp8, float kv_scale,
                      int num_pages, int page_size, const int32_t* block_table, int R,
                      int q_per_req, int max_pages_per_req, const int32_t* kv_bounds,
                      const void* gate, int gate_dim, int H, float softmax_scale, int num_splits,
                      int form, void* workspace, size_t workspace_bytes, void* out, float* lse,
                      int32_t* status, sv_stream_t stream, uint64_t wait_ns = kWaitTimeoutNs) {
  if (R < 0 || q_per_req < 1 || H < 1 || max_pages_per_req < 0 || num_pages < 0)
    return SV_ERR_SHAPE;
  if (gate_dim != kD && gate_dim != 1) return SV_ERR_UNSUPPORTED;
  if (!valid_form(form)) return SV_ERR_UNSUPPORTED;
  if (page_size != SV_PAGE_SIZE) return SV_ERR_UNSUPPORTED;
  if ((num_splits < 0 && num_splits != SV_SPLITS_BALANCED && num_splits != SV_SPLITS_WAVE) ||
      num_splits > SV_MAX_SPLITS)
    return SV_ERR_SHAPE;
  if (num_splits == SV_SPLITS_BALANCED && max_pages_per_req > 0xFFFF) return SV_ERR_SHAPE;
  const long long T = (long long)R * q_per_req;
  if (T == 0) return SV_OK;
  if (T * H > 0x7FFFFFFFll || (long long)num_pages * kTileN > 0x7FFFFFFFll) return SV_ERR_SHAPE;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return SV_ERR_SHAPE;
  if (kv_fp8 && (!(kv_scale > 0.f) || !std::isfinite(kv_scale))) return SV_ERR_SHAPE;
  if (num_pages < 1 || max_pages_per_req < 1) return SV_ERR_SHAPE;
  if (!q_latent || !kv_pages || !block_table || !kv_bounds || !gate || !out || !lse)
    return SV_ERR_NULL;
  if (misaligned(q_latent, 16) || misaligned(kv_pages, 16) || misaligned(gate, 16) ||
      misaligned(out, 16) || misaligned(lse, 4) || misaligned(block_table, 4) ||
      misaligned(kv_bounds, 4))
    return SV_ERR_ALIGN;
  if ((num_splits == SV_SPLITS_BALANCED || num_splits > 1) && !workspace) return SV_ERR_WORKSPACE;
  int sm_count = 0;
  if (!device_setup(&sm_count)) return SV_ERR_DEVICE;
  const int S = num_splits != 0 ? num_splits
                                : sv_mla_verify_num_splits(R, q_per_req, H, max_pages_per_req, form);
  const bool balanced = (S == SV_SPLITS_BALANCED);
  const bool wave = (S == SV_SPLITS_WAVE);
  const long long Mq_ll = (long long)H * q_per_req;
  const int n_mt = (int)((Mq_ll + kMTile - 1) / kMTile);
  int wave_k = 0, wave_s = 0;
  if (wave && !wave_params(R, n_mt, max_pages_per_req, sm_count, &wave_k, &wave_s)) return SV_ERR_SHAPE;
  const long long wave_slots = (long long)(R - wave_k) * wave_s;
  // stacked instance: requests of <= 64 query rows, uniform splits or the
  // balanced plan; its row maps have 64-row boxes
  const bool stack = !wave && (balanced ? use_stack_balanced(Mq_ll, form)
                                        : use_stack(Mq_ll, max_pages_per_req, S, form));
  __nv_bfloat16* part_o = nullptr;
  float* part_lse = nullptr;
  PlanLayout PL{};
  char* plan_base_ptr = nullptr;
  if (balanced) {
    if (!workspace) return SV_ERR_WORKSPACE;
    if (misaligned(workspace, 256)) return SV_ERR_ALIGN;
    PL = plan_layout(R, (int)Mq_ll, n_mt, sm_count, stack);
    if (workspace_bytes < PL.total ||
        workspace_bytes < sv_mla_verify_workspace_bytes((int)T, H, SV_SPLITS_BALANCED))
      return SV_ERR_WORKSPACE;
    plan_base_ptr = static_cast<char*>(workspace);
    part_o = reinterpret_cast<__nv_bfloat16*>(plan_base_ptr + PL.part_o);
    part_lse = reinterpret_cast<float*>(plan_base_ptr + PL.part_lse);
  } else if (wave) {
    if (!workspace) return SV_ERR_WORKSPACE;
    if (misaligned(workspace, 256)) return SV_ERR_ALIGN;
    if (workspace_bytes < sv_mla_verify_workspace_bytes((int)T, H, SV_SPLITS_WAVE)) return SV_ERR_WORKSPACE;
    part_o = static_cast<__nv_bfloat16*>(workspace);
    part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        align256((size_t)wave_slots * Mq_ll * kD * sizeof(__nv_bfloat16)));
  } else if (S > 1) {
    if (!workspace) return SV_ERR_WORKSPACE;
    if (misaligned(workspace, 256)) return SV_ERR_ALIGN;
    if (workspace_bytes < sv_mla_verify_workspace_bytes((int)T, H, S)) return SV_ERR_WORKSPACE;
    part_o = static_cast<__nv_bfloat16*>(workspace);
    part_lse = reinterpret_cast<float*>(part_o + (size_t)S * T * H * kD);
  }
  if (!get_encode_fn()) return SV_ERR_DEVICE;
  const long long Mq = (long long)H * q_per_req;
  const int m_box = stack ? 64 : kMTile;
  CUtensorMap tmap_kv, tmap_q, tmap_gate, tmap_out, tmap_part;
  {
    const cuuint64_t kv_dims[2] = {(cuuint64_t)kD, (cuuint64_t)num_pages * kTileN};
    const cuuint32_t kv_box[2] = {64, (cuuint32_t)kTileN};
    const cuuint64_t row_dims[3] = {(cuuint64_t)kD, (cuuint64_t)Mq, (cuuint64_t)R};
    const cuuint32_t row_box[3] = {64, (cuuint32_t)m_box, 1};
    const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // fp8 KV is read by the converter warps, not through a tensor map
    if ((kv_fp8 ? !encode_map(&tmap_kv, bf16, 2, q_latent, 3, row_dims, row_box)
                : !encode_map(&tmap_kv, bf16, 2, kv_pages, 2, kv_dims, kv_box)) ||
        !encode_map(&tmap_q, bf16, 2, q_latent, 3, row_dims, row_box) ||
        (gate_dim == kD ? !encode_map(&tmap_gate, bf16, 2, gate, 3, row_dims, row_box)
                        : !encode_map(&tmap_gate, bf16, 2, q_latent, 3, row_dims, row_box)) ||
        !encode_map(&tmap_out, bf16, 2, out, 3, row_dims, row_box))
      return SV_ERR_ALIGN;
    if (balanced || wave) {
      const cuuint64_t slots = balanced ? (cuuint64_t)PL.slots_max : (cuuint64_t)wave_slots;
      const cuuint64_t part_dims[4] = {(cuuint64_t)kD, (cuuint64_t)Mq, 1, slots};
      const cuuint32_t part_box[4] = {64, (cuuint32_t)m_box, 1, 1};
      if (!encode_map(&tmap_part, bf16, 2, part_o, 4, part_dims, part_box))
        return SV_ERR_ALIGN;
    } else if (S > 1) {
      const cuuint64_t part_dims[4] = {(cuuint64_t)kD, (cuuint64_t)Mq, (cuuint64_t)R, (cuuint64_t)S};
      const cuuint32_t part_box[4] = {64, (cuuint32_t)m_box, 1, 1};
      if (!encode_map(&tmap_part, bf16, 2, part_o, 4, part_dims, part_box))
        return SV_ERR_ALIGN;
    } else {
      tmap_part = tmap_out;  // unused with one split
    }
  }

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
  prm.n_mtiles = n_mt;
  prm.scale_log2 = softmax_scale * 1.4426950408889634f;
  prm.units = nullptr;
  prm.plan_header = nullptr;
  prm.part_w_stride = T * H;
  prm.gate_dim = gate_dim;
  prm.kv_scale = kv_fp8 ? kv_scale : 1.0f;
  prm.kv8 = kv_fp8 ? static_cast<const uint8_t*>(kv_pages) : nullptr;
  prm.wave_k = 0;
  prm.wave_s = 0;
  prm.wait_ns = wait_ns;
  prm.part_lse_entries = balanced ? (long long)PL.slots_max * Mq_ll
                         : wave   ? wave_slots * Mq_ll
                                  : (S > 1 ? (long long)S * T * H : 0);
  prm.wave_k = wave_k;
  prm.wave_s = wave_s;
  // fp8: the pool scale multiplies every score (folded into the scale here)
  // and the output (applied in the epilogue)
  if (kv_fp8) prm.scale_log2 *= kv_scale;
  // long units (uniform splits of >= kTwoIssuerTiles tiles, the balanced
  // plan's pieces, the wave mode's whole requests) take the instance with a
  // second score issuer (a unit with fewer tiles runs on one issuer in it)
  const bool two = balanced || wave || ((long long)max_pages_per_req + S - 1) / S >= kTwoIssuerTiles;
  const bool short_waits = wait_ns < kWaitTimeoutNs;
  const VerifyKernel kernel =
      kVerifyKernels[(kv_fp8 ? 1 : 0) | (two ? 2 : 0) | (stack ? 4 : 0) | (short_waits ? 8 : 0)];
  const int threads = kv_fp8 ? (two ? KernelShape<true, true>::kThreads : KernelShape<true, false>::kThreads)
                             : (two ? KernelShape<false, true>::kThreads : KernelShape<false, false>::kThreads);
  const int smem = KernelShape<false, false>::kSmemBytes;  // the same for every instance
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  if (wave) {
    prm.part_w_stride = Mq_ll;
    const long long ctas = 2ll * n_mt * (wave_k + wave_slots);
    kernel<<<(unsigned)ctas, threads, smem, st>>>(tmap_kv, tmap_q, tmap_gate, tmap_out, tmap_part, prm);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_LAUNCH;
    // merge only the rows of the split requests
    if (launch_lse_combine(part_o, true, part_lse, wave_s, T * H, gate, out, lse, st, nullptr, nullptr,
                           (int)Mq_ll, gate_dim, (long long)wave_k * Mq_ll, wave_k) != cudaSuccess)
      return SV_ERR_LAUNCH;
    return SV_OK;
  }
  if (!balanced) {
    const long long ctas = (stack ? 1ll : 2ll) * R * prm.n_mtiles * S;
    if (ctas > 0x7FFFFFFFll) return SV_ERR_SHAPE;
    kernel<<<(unsigned)ctas, threads, smem, st>>>(tmap_kv, tmap_q, tmap_gate, tmap_out, tmap_part,
                                                  prm);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_LAUNCH;
    if (S > 1 && launch_lse_combine(part_o, true, part_lse, S, T * H, gate, out, lse, st, nullptr,
                                    nullptr, 1, gate_dim) != cudaSuccess)
      return SV_ERR_LAUNCH;
    return SV_OK;
  }

  // balanced plan: plan kernel, then the attention kernel and the merge, each
  // a programmatic dependent launch of the one before
  int* header = reinterpret_cast<int*>(plan_base_ptr);
  int* splits = reinterpret_cast<int*>(plan_base_ptr + PL.splits);
  int* pbase = reinterpret_cast<int*>(plan_base_ptr + PL.base);
  int4* units = reinterpret_cast<int4*>(plan_base_ptr + PL.units);
  plan_kernel<<<1, kPlanThreads, 0, st>>>(kv_bounds, R, q_per_req, max_pages_per_req,
                                          stack ? 1 : 2 * n_mt, stack ? 1 : n_mt, stack ? kStackPlanDiv : 1, sm_count,
                                          PL.units_max, PL.slots_max, header, splits, pbase, units,
                                          status);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_LAUNCH;
  prm.units = units;
  prm.plan_header = header;
  prm.part_w_stride = Mq_ll;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)PL.units_max, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, tmap_kv, tmap_q, tmap_gate, tmap_out, tmap_part,
                         prm) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_LAUNCH;
  }
  if (launch_lse_combine(part_o, true, part_lse, 0, T * H, gate, out, lse, st, splits, pbase,
                         (int)Mq_ll, gate_dim) != cudaSuccess)
    return SV_ERR_LAUNCH;
  return SV_OK;
}
}  // namespace
}  // namespace sv

extern "C" sv_status mla_verify_decode_gated(const void* q_latent, const void* kv_pages,
                                             int num_pages, int page_size,
                                             const int32_t* block_table, int R, int q_per_req,
                                             int max_pages_per_req, const int32_t* kv_bounds,
                                             const void* gate, int gate_dim, int H,
                                             float softmax_scale, int num_splits, int form,
                                             void* workspace, size_t workspace_bytes, void* out,
                                             float* lse, int32_t* status, sv_stream_t stream) {
  return sv::verify_impl(q_latent, kv_pages, false, 1.0f, num_pages, page_size, block_table, R,
                         q_per_req, max_pages_per_req, kv_bounds, gate, gate_dim, H,
                         softmax_scale, num_splits, form, workspace, workspace_bytes, out, lse,
                         status, stream);
}

extern "C" sv_status mla_verify_decode_kv8(const void* q_latent, const void* kv_pages_e4m3,
                                           float kv_scale, int num_pages, int page_size,
                                           const int32_t* block_table, int R, int q_per_req,
                                           int max_pages_per_req, const int32_t* kv_bounds,
                                           const void* gate, int gate_dim, int H,
                                           float softmax_scale, int num_splits, int form,
                                           void* workspace, size_t workspace_bytes, void* out,
                                           float* lse, int32_t* status, sv_stream_t stream) {
  return sv::verify_impl(q_latent, kv_pages_e4m3, true, kv_scale, num_pages, page_size,
                         block_table, R, q_per_req, max_pages_per_req, kv_bounds, gate, gate_dim,
                         H, softmax_scale, num_splits, form, workspace, workspace_bytes, out, lse,
                         status, stream);
}

// Test entry point: the verify attention (bf16 KV, or e4m3 codes with
// kv_fp8 != 0 and their scale) with the limit of every bounded wait of the
// attention kernel lowered to wait_ns (the drains at teardown keep theirs).
extern "C" sv_status sv_test_mla_verify_decode_wait_limit(
    const void* q_latent, const void* kv_pages, int kv_fp8, float kv_scale, int num_pages, int page_size,
    const int32_t* block_table, int R, int q_per_req, int max_pages_per_req, const int32_t* kv_bounds,
    const void* gate, int gate_dim, int H, float softmax_scale, int num_splits, int form, void* workspace,
    size_t workspace_bytes, void* out, float* lse, int32_t* status, sv_stream_t stream, uint64_t wait_ns) {
  if (wait_ns > sv::kWaitTimeoutNs) return SV_ERR_SHAPE;  // it only shortens the waits
  return sv::verify_impl(q_latent, kv_pages, kv_fp8 != 0, kv_fp8 ? kv_scale : 1.0f, num_pages, page_size,
                         block_table, R, q_per_req, max_pages_per_req, kv_bounds, gate, gate_dim, H,
                         softmax_scale, num_splits, form, workspace, workspace_bytes, out, lse, status, stream,
                         wait_ns);
}

extern "C" sv_status mla_verify_decode(const void* q_latent, const void* kv_pages, int num_pages,
                                       int page_size, const int32_t* block_table, int R,
                                       int q_per_req, int max_pages_per_req,
                                       const int32_t* kv_bounds, const void* gate, int H,
                                       float softmax_scale, int num_splits, void* workspace,
                                       size_t workspace_bytes, void* out, float* lse,
                                       int32_t* status, sv_stream_t stream) {
  return mla_verify_decode_gated(q_latent, kv_pages, num_pages, page_size, block_table, R,
                                 q_per_req, max_pages_per_req, kv_bounds, gate, SV_LATENT_DIM, H,
                                 softmax_scale, num_splits, SV_FORM_AUTO, workspace,
                                 workspace_bytes, out, lse, status, stream);
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
