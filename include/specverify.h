/*
 * specverify.h - C ABI of the GB300 (sm_103a) speculative-decoding verify step
 * for absorbed, gated NoPE MLA over a paged bf16 latent KV cache.
 *
 * One verify step: each of R requests feeds a verify group of 1 target token
 * plus k drafted tokens ("M* PR #257: Kimi K3 support with DSpark speculative
 * decoding", section "Speculative decoding").  T = R*(k+1) query tokens,
 * H heads, latent width D = 512.
 *
 *   mla_verify_decode   attention of every token over its request's paged
 *                       latent rows, bounded per token, split over KV, with
 *                       the LSE merge and the sigmoid gate fused in.
 *   mla_lse_combine     the LSE merge + gate of split partials on its own.
 *   mla_verify_decode_gated  the same with a head-wise ([T][H]) gate.
 *   mla_verify_decode_kv8    the same over an fp8 (E4M3 + scale) page pool.
 *   mla_wuv_project     the per-head W_UV value up-projection after the merge.
 *   mla_kv_append       the verify tokens' latent rows into the paged cache.
 *   spec_verify_sampled rejection-sampling verification (probabilistic drafts).
 *   spec_verify_greedy  target argmax, accepted draft prefix, next token and
 *                       trimmed per-request KV length.
 *
 * Conventions shared by every call:
 *  - Every pointer named "device" is CUDA device memory owned by the caller;
 *    the library never allocates, never frees and never synchronises the host.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).
 *  - Host-side argument checks run before any launch; a failed check returns
 *    its sv_status code and launches nothing.
 *  - Bad *device data* (a block-table entry outside the pool, a bound outside
 *    [0, max_pages_per_req*page_size]) never traps: the kernel ORs an
 *    SV_DEV_* bit into the caller's device status word, substitutes a safe
 *    value (page 0, the clamped bound) and carries on; the outputs of that
 *    call are then undefined.  The caller reads the status word.
 *  - Every wait inside a kernel is bounded (about two seconds); a wait that
 *    gives up ORs SV_DEV_TIMEOUT into the status word and the kernel returns.
 */
#ifndef SPECVERIFY_H_
#define SPECVERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sv_stream_t; /* a cudaStream_t */

typedef enum {
  SV_OK = 0,
  SV_ERR_NULL = 1,        /* a required pointer is NULL                       */
  SV_ERR_SHAPE = 2,       /* a size is negative or inconsistent               */
  SV_ERR_ALIGN = 3,       /* a pointer misses its required alignment          */
  SV_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required       */
  SV_ERR_UNSUPPORTED = 5, /* valid but unsupported (page_size != 64, D != 512) */
  SV_ERR_LAUNCH = 6,      /* the CUDA launch itself failed                    */
  SV_ERR_DEVICE_DATA = 7, /* reserved for callers mapping SV_DEV_* bits       */
  SV_ERR_TIMEOUT = 8,     /* reserved for callers mapping SV_DEV_TIMEOUT      */
  SV_ERR_DEVICE = 9       /* no usable sm_103a device / attribute query failed */
} sv_status;

/* bits ORed into the device status word */
#define SV_DEV_BAD_PAGE  0x1  /* block_table entry < 0 or >= num_pages was needed */
#define SV_DEV_BAD_BOUND 0x2  /* kv_bounds[t] < 0 or > max_pages_per_req*page_size */
#define SV_DEV_TIMEOUT   0x4  /* a bounded in-kernel wait gave up                 */
/* only in the index-checking debug build (compiled with -DSPECVERIFY_DEBUG):
 * an index or address check failed and its access was skipped */
#define SV_DEV_DEBUG_CHECK 0x8

#define SV_LATENT_DIM 512
#define SV_PAGE_SIZE 64
#define SV_MAX_SPLITS 64
/* num_splits value selecting the balanced split plan (see mla_verify_decode). */
#define SV_SPLITS_BALANCED (-1)
/* num_splits value selecting the wave split mode (see mla_verify_decode). */
#define SV_SPLITS_WAVE (-2)

/* Human-readable name of a status code (static string, never NULL). */
const char* sv_status_string(sv_status s);

/* ------------------------------------------------------------------------
 * mla_verify_decode
 *
 * Absorbed, gated NoPE MLA decode attention for verify groups ("M* PR #257",
 * section "Model": gated NoPE MLA with absorbed projections), with the
 * per-token attention bound, the widened masked span and the (-inf, 0)
 * stats identity of "TensorRT-LLM PR #18166: Kimi K3 DSpark speculative
 * decoding under Helix CP" (first commit message and Summary).
 *
 * For token t (request r = t / q_per_req) and head h, with b = kv_bounds[t]
 * and c_j the latent row of KV position j (page block_table[r][j/64], slot
 * j%64):
 *     s_j  = softmax_scale * <q[t][h], c_j>              for j < b
 *     lse  = ln sum_j exp(s_j)                           (-inf when b == 0)
 *     o    = sum_j exp(s_j - lse) * c_j                  (0    when b == 0)
 *     out  = sigmoid(gate[t][h]) * o   (elementwise over the 512 columns)
 * The k+1 tokens of a request are folded into M = H*(k+1) query rows that
 * share the request's KV (row = t_local*H + h), processed as 128-row tiles;
 * each (row tile, KV split) runs on two CTAs, one per 256-column latent half
 * of the output.  With uniform splits and M <= 64, one CTA may hold both
 * halves instead (the "stacked" form, see SV_FORM_* below); this call takes
 * the automatic choice (SV_FORM_AUTO).
 *
 * Arguments (all device pointers unless stated):
 *   q_latent      bf16 [T][H][512], 16-byte aligned, contiguous.
 *   kv_pages      bf16 [num_pages][page_size][512], 16-byte aligned
 *                 (the page pool; read through a TMA tensor map).
 *   num_pages     pool size in pages (>= 1 when any bound is > 0).
 *   page_size     must be 64 (else SV_ERR_UNSUPPORTED).
 *   block_table   int32 [R][max_pages_per_req]: page ids; entries past a
 *                 request's last needed page are never read.
 *   R, q_per_req  requests and tokens per request (k+1 >= 1); T = R*q_per_req.
 *   kv_bounds     int32 [T]: token t sees positions j < kv_bounds[t];
 *                 0 <= kv_bounds[t] <= max_pages_per_req*page_size.
 *   gate          bf16 [T][H][512].
 *   H             heads, >= 1.
 *   softmax_scale scale of the scores (finite, > 0).
 *   num_splits    how the KV of each request is cut into work units:
 *                 1..SV_MAX_SPLITS: S uniform splits per (request, row tile);
 *                   split s of request r covers KV tiles
 *                   [s*n_r/S, (s+1)*n_r/S) (integer division) with
 *                   n_r = ceil(max_t kv_bounds[t] / 64) over r's tokens.
 *                 SV_SPLITS_BALANCED (-1): a plan computed on the device from
 *                   kv_bounds cuts every request into pieces of c pages,
 *                   c = max(ceil(sum_r n_r * n_tiles / SMs), ceil(max_r n_r / 64))
 *                   (n_tiles = 128-row tiles per request; two CTAs per
 *                   128-row tile and piece: about two CTAs per SM), or in
 *                   the stacked form (one CTA per piece)
 *                   c = max(ceil(sum_r n_r / SMs), ceil(max_r n_r / 64)), so
 *                   that requests of very different lengths give the SMs
 *                   equal work; the pieces run longest first.  One extra
 *                   small kernel.  A plan that does not fit the workspace
 *                   sets SV_DEV_BAD_BOUND and computes nothing.
 *                 SV_SPLITS_WAVE (-2): for batches whose 2 * n_tiles * R
 *                   CTAs fill the SMs more than once but less than twice:
 *                   requests 0..k-1 are not split and fill the first wave,
 *                   each other request is cut into s uniform pieces that
 *                   fill the second, with k = floor(SMs / (2 n_tiles)) and
 *                   s = max(2, floor(SMs / (2 n_tiles (R - k)))) (at most
 *                   max_pages_per_req / 2); SV_ERR_SHAPE where that does not
 *                   apply.  The merge kernel then reads only the split
 *                   requests' rows.
 *                 0: automatic (sv_mla_verify_num_splits).
 *                 The result does not depend on the choice beyond rounding.
 *   workspace     device scratch of at least
 *                 sv_mla_verify_workspace_bytes(T, H, S) bytes (S = the
 *                 num_splits used, after resolving 0), 256-byte aligned; may
 *                 be NULL when S == 1.  With 2..SV_MAX_SPLITS uniform splits
 *                 it holds the split partials: part_o bf16 [S][T][H][512]
 *                 (round to nearest even) followed by part_lse fp32
 *                 [S][T][H] (lse of the split's KV range, natural log, -inf
 *                 for an empty range; part_o normalised within the split, 0
 *                 for an empty range).  With the balanced plan its layout is
 *                 internal.
 *   workspace_bytes  its size in bytes.
 *   out           bf16 [T][H][512] (round to nearest even).
 *   lse           fp32 [T][H], natural log of the ungated scaled scores.
 *   status        device int32, ORed with SV_DEV_* bits; may be NULL.
 *   stream        CUDA stream.
 * Returns SV_OK after enqueueing, or the first failed check.
 * ---------------------------------------------------------------------- */
/* The kernel form of the attention call, chosen per call (the `form`
 * argument of mla_verify_decode_gated / _kv8 and sv_mla_verify_num_splits;
 * mla_verify_decode uses SV_FORM_AUTO).  The stacked form runs requests of
 * M = H*q_per_req <= 64 query rows with uniform splits or the balanced plan
 * on one CTA per (request, split or piece): rows 64..127 of the CTA's
 * 128-row MMA tile repeat rows
 * 0..63, and the softmax weights P form a block-diagonal operand over the KV
 * tile taken twice, so TMEM lanes 0..63 accumulate latent columns 0..255 and
 * lanes 64..127 columns 256..511 (no second CTA recomputing the scores).
 * The result is the same beyond rounding.
 *   SV_FORM_AUTO      the stacked form when M <= 64 and either the
 *                     balanced plan runs or the splits are uniform and a
 *                     unit holds at least 4 KV tiles
 *                     (ceil(max_pages_per_req / S) >= 4); else two CTAs.
 *   SV_FORM_TWO_CTA   always two CTAs per unit, one per latent half.
 *   SV_FORM_STACKED   the stacked form whenever M <= 64 and the splits are
 *                     uniform or balanced (else two CTAs).
 * Any other value: SV_ERR_UNSUPPORTED (sv_mla_verify_num_splits returns 0). */
#define SV_FORM_AUTO 0
#define SV_FORM_TWO_CTA 1
#define SV_FORM_STACKED 2

/* The num_splits that 0 resolves to on the current device for the given
 * form (it only looks at the sizes, never at device data):
 * SV_SPLITS_BALANCED when R >= 2, max_pages_per_req >= 64 and
 * 2 * ceil(H*q_per_req/128) * R <= SMs (long contexts whose units fit the SMs
 * once); SV_SPLITS_WAVE when those CTAs fill the SMs more than once but less
 * than twice (and the stacked form is not taken); else a uniform count that
 * fills the SMs once with >= 2 KV tiles per split, counting one CTA per
 * (request, row tile, split) when the stacked form will be taken for it and
 * two otherwise.  The same count serves the
 * fp8 entry point.  sv_mla_verify_workspace_bytes accepts any num_splits
 * value mla_verify_decode accepts except 0 (resolve it first). */
int sv_mla_verify_num_splits(int R, int q_per_req, int H, int max_pages_per_req, int form);
size_t sv_mla_verify_workspace_bytes(int T, int H, int num_splits);

sv_status mla_verify_decode(const void* q_latent, const void* kv_pages, int num_pages,
                            int page_size, const int32_t* block_table, int R, int q_per_req,
                            int max_pages_per_req, const int32_t* kv_bounds, const void* gate,
                            int H, float softmax_scale, int num_splits, void* workspace,
                            size_t workspace_bytes, void* out, float* lse, int32_t* status,
                            sv_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_verify_decode_gated
 *
 * mla_verify_decode with a choice of gate shape (the head-wise form is the
 * "next" variant for the H = 96 Kimi K3 configuration of "TensorRT-LLM PR
 * #18166"; only a gate that is constant over a head's latent row commutes
 * with the later per-head W_UV projection):
 *   gate_dim == 512: gate bf16 [T][H][512], out = sigmoid(gate) * o
 *                    elementwise (exactly mla_verify_decode);
 *   gate_dim == 1:   gate bf16 [T][H], out[t][h][:] = sigmoid(gate[t][h]) * o.
 * Any other gate_dim returns SV_ERR_UNSUPPORTED.  `form` picks the kernel
 * form (SV_FORM_*; num_splits = 0 then resolves to
 * sv_mla_verify_num_splits(..., form)).  All other arguments, layouts and
 * errors as mla_verify_decode; gate must be 16-byte aligned.
 * ---------------------------------------------------------------------- */
sv_status mla_verify_decode_gated(const void* q_latent, const void* kv_pages, int num_pages,
                                  int page_size, const int32_t* block_table, int R,
                                  int q_per_req, int max_pages_per_req, const int32_t* kv_bounds,
                                  const void* gate, int gate_dim, int H, float softmax_scale,
                                  int num_splits, int form, void* workspace,
                                  size_t workspace_bytes, void* out, float* lse, int32_t* status,
                                  sv_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_verify_decode_kv8
 *
 * mla_verify_decode_gated over an fp8 latent KV cache (the fp8 KV deployment
 * on the model card "RedHatAI/Kimi-K3-speculator.dspark", section
 * "Deployment"; the verify kernel of "TensorRT-LLM PR #18166" rejects fp8 KV,
 * so this is the "next" variant): kv_pages_e4m3 holds OCP FP8 E4M3 codes
 * [num_pages][64][512] (1 byte each, 16-byte aligned) and the cached latent
 * row is code value * kv_scale (one scale for the pool, finite and > 0).
 * The tensor-core products of this variant take f16 operands: each KV tile
 * is converted to f16 in shared memory (exact), q_latent is rounded to f16
 * (exact for |q| in [2^-14, 65504]; larger magnitudes overflow, so q must
 * stay below 65504) and the softmax weights P are f16 (bf16 in the bf16
 * variant); kv_scale is folded into the score scale and the output.
 * Everything else as mla_verify_decode_gated; the workspace query is the
 * same.
 * ---------------------------------------------------------------------- */
sv_status mla_verify_decode_kv8(const void* q_latent, const void* kv_pages_e4m3, float kv_scale,
                                int num_pages, int page_size, const int32_t* block_table, int R,
                                int q_per_req, int max_pages_per_req, const int32_t* kv_bounds,
                                const void* gate, int gate_dim, int H, float softmax_scale,
                                int num_splits, int form, void* workspace,
                                size_t workspace_bytes, void* out, float* lse, int32_t* status,
                                sv_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_wuv_project
 *
 * Per-head value up-projection of the absorbed attention output, the
 * "LSE combine + W_UV" step after the merge (vLLM page
 * "kimi_k3/nvidia/specialized_decode/drafter/model"):
 *     out_v[t][h][j] = sum_d w_uv[h][j][d] * x[t][h][d]     (fp32 accumulate)
 *
 *   x       bf16 [T][H][512] (e.g. the out of mla_verify_decode), 16-byte
 *           aligned.
 *   w_uv    bf16 [H][v_dim][512], 16-byte aligned.
 *   v_dim   a multiple of 32 in [32, 256] (else SV_ERR_UNSUPPORTED).
 *   out_v   bf16 [T][H][v_dim] (round to nearest even), 16-byte aligned.
 *   status  device int32 ORed with SV_DEV_TIMEOUT if a bounded wait gives
 *           up; may be NULL.
 * One tcgen05 GEMM per (head, 128-token tile) on `stream`.
 * ---------------------------------------------------------------------- */
sv_status mla_wuv_project(const void* x, const void* w_uv, int T, int H, int v_dim, void* out_v,
                          int32_t* status, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_kv_append
 *
 * Writes the latent KV rows of the verify tokens into the paged cache before
 * the attention reads them: the NoPE counterpart of the per-token KV write
 * slot of "TensorRT-LLM PR #18166: Kimi K3 DSpark speculative decoding under
 * Helix CP" (first commit message: global position -> write slot, -1 = not
 * owned; on one GPU every position is owned).
 *
 * Token t (request r = t / q_per_req) with positions[t] = pos >= 0 stores
 * kv_new[t] in page block_table[r][pos / 64], slot pos % 64; pos = -1 skips
 * the token.  Positions of one call must be distinct per request.
 *
 *   kv_new       bf16 [T][512], 16-byte aligned (T = R*q_per_req).
 *   positions    int32 [T].
 *   block_table  int32 [R][max_pages_per_req].
 *   kv_pages     bf16 [num_pages][page_size][512], 16-byte aligned, updated
 *                in place.
 *   page_size    must be 64.
 *   status       device int32, ORed with SV_DEV_BAD_BOUND (pos past the
 *                table) or SV_DEV_BAD_PAGE (entry outside the pool); such a
 *                token is skipped.  May be NULL.
 * ---------------------------------------------------------------------- */
sv_status mla_kv_append(const void* kv_new, const int32_t* positions, const int32_t* block_table,
                        int R, int q_per_req, int max_pages_per_req, void* kv_pages,
                        int num_pages, int page_size, int32_t* status, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_lse_combine
 *
 * Merge of split-KV partials by their log-sum-exp (the CP / DCP LSE merge of
 * "TensorRT-LLM PR #18166", second and third commit messages, and of the vLLM
 * page "kimi_k3/nvidia/specialized_decode/drafter/model", DraftDcp), plus the
 * sigmoid-gate epilogue:
 *     lse = ln sum_s exp(part_lse[s])
 *     o   = sum_s exp(part_lse[s] - lse) * part_o[s]
 *     out = sigmoid(gate) * o
 * A row whose partials are all -inf gives lse = -inf and out = 0 (never NaN).
 *
 *   part_o    fp32 [S][T][H][512], 16-byte aligned.
 *   part_lse  fp32 [S][T][H].
 *   S         1..SV_MAX_SPLITS;  T, H >= 0.
 *   gate      bf16 [T][H][512], 8-byte aligned.
 *   out       bf16 [T][H][512], 8-byte aligned;  lse fp32 [T][H].
 * ---------------------------------------------------------------------- */
sv_status mla_lse_combine(const float* part_o, const float* part_lse, int S, int T, int H,
                          const void* gate, void* out, float* lse, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * spec_verify_greedy
 *
 * Greedy verification with KV trim ("M* PR #257", section "Speculative
 * decoding": verification is greedy, the KV trims rejected tails):
 *     a[t]          = argmax_v logits[t][v]     (lowest v on ties; -0 == +0)
 *     accepted[r]   = n = largest m <= k with draft_tokens[r][j-1] == a[r*(k+1)+j-1]
 *                     for every j = 1..m
 *     next_tokens[r]= a[r*(k+1) + n]
 *     kv_lens_out[r]= kv_lens_in[r] - (k - n)
 * kv_lens_in counts the k+1 verify tokens already written to the cache.
 *
 *   logits        fp32 [T][V], T = R*(k+1), V >= 1; values must be finite.
 *   draft_tokens  int32 [R][k] (may be NULL when k == 0).
 *   kv_lens_in    int32 [R].
 *   argmax_ids    int32 [T]; accepted, next_tokens, kv_lens_out int32 [R].
 *   workspace     device scratch of sv_greedy_workspace_bytes(T, V) bytes,
 *                 256-byte aligned.  It must be zero-filled before its first
 *                 use (e.g. cudaMemsetAsync); every call leaves it zero-filled
 *                 again, so one zeroing serves any number of later calls on
 *                 the same stream.  Calls sharing one workspace must not run
 *                 concurrently.
 * ---------------------------------------------------------------------- */
size_t sv_greedy_workspace_bytes(int T, int V);

sv_status spec_verify_greedy(const float* logits, int T, int V, int R, int k,
                             const int32_t* draft_tokens, const int32_t* kv_lens_in,
                             int32_t* argmax_ids, int32_t* accepted, int32_t* next_tokens,
                             int32_t* kv_lens_out, void* workspace, size_t workspace_bytes,
                             sv_stream_t stream);

/* ------------------------------------------------------------------------
 * spec_verify_sampled
 *
 * Sampled verification with KV trim ("M* PR #257", section "Speculative
 * decoding": verification is greedy or sampled, FlashInfer's chain sampling;
 * the model card "RedHatAI/Kimi-K3-speculator.dspark", section "Deployment",
 * draws the drafts probabilistically).  The pages give no formula; this is
 * token-wise chain rejection sampling (speculative sampling, Leviathan et al.
 * 2023; Chen et al. 2023):
 *     p_t        = softmax(logits[t] / temperature),  t = r*(k+1) + j
 *     draft j    accepted iff uniforms[r][j] * q(d) < p_t(d),
 *                d = draft_tokens[r][j], q = draft_probs[r][j]
 *                (a draft id outside [0, V) is rejected)
 *     accepted[r]   = n = number of drafts before the first rejection
 *     next_tokens[r]= draw from max(0, p_t - q) at the first rejection
 *                     (p_t if that is zero everywhere), or from p of token
 *                     r*(k+1)+k when all k are accepted; a draw from weights
 *                     w with u = uniforms[r][k] is the smallest v with
 *                     sum_{i<=v} w_i > u * sum(w)
 *     kv_lens_out[r]= kv_lens_in[r] - (k - n)
 * Arithmetic is fp32 on the device: a decision whose margin is within fp32
 * rounding (|u*q - p| ~ 1e-6 relative, or u*W within ~1e-5 W of a CDF step)
 * may fall either way.
 *
 *   logits        fp32 [R*(k+1)][V], finite, V >= 1.
 *   temperature   > 0 and finite; logits / temperature must stay finite.
 *   draft_tokens  int32 [R][k];  draft_probs fp32 [R][k][V] (each row the
 *                 distribution its draft was drawn from).  Both may be NULL
 *                 when k == 0.
 *   uniforms      fp32 [R][k+1] in [0, 1): the caller's random numbers.
 *   kv_lens_in    int32 [R];  accepted, next_tokens, kv_lens_out int32 [R].
 *   workspace     sv_sampled_workspace_bytes(R, k, V) bytes, 256-byte
 *                 aligned, zero-filled before its first use; every call leaves
 *                 its counters zero again.  Calls sharing one workspace must
 *                 not run concurrently.
 * Two kernels on `stream` (the second a programmatic dependent launch).
 * ---------------------------------------------------------------------- */
size_t sv_sampled_workspace_bytes(int R, int k, int V);

sv_status spec_verify_sampled(const float* logits, int R, int k, int V, float temperature,
                              const int32_t* draft_tokens, const float* draft_probs,
                              const float* uniforms, const int32_t* kv_lens_in,
                              int32_t* accepted, int32_t* next_tokens, int32_t* kv_lens_out,
                              void* workspace, size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------
 * spec_verify_greedy_noalloc
 *
 * The paper has no counterpart to this call: it is an addition for callers
 * that cannot allocate device memory when they verify (for example a serving
 * engine that has reserved nearly all HBM for its own KV-cache pool, or a
 * plugin whose host framework owns the device allocator) and so cannot pass
 * the workspace spec_verify_greedy needs.
 *
 * Same arguments, results and errors as spec_verify_greedy, without the
 * workspace.  The scratch lives in a file-scope device array of 512 KiB that
 * every GPU loading this library keeps until the process exits.
 *  - A problem with sv_greedy_workspace_bytes(T, V) > 512 KiB is rejected with
 *    SV_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device looks up the array's address with that device
 *    current; make that first call before any stream capture begins.
 *  - Each call clears the part of the array it uses (the counter and the
 *    per-row keys: 256 + 8 T bytes) with cudaMemsetAsync on `stream`
 *    before its kernel; nothing is allocated or freed.
 *  - All calls share the one array: calls whose kernels may overlap on the
 *    GPU (unordered streams, several host threads) race and give wrong
 *    results.  Calls in order on one stream are safe.
 * ---------------------------------------------------------------------- */
sv_status spec_verify_greedy_noalloc(const float* logits, int T, int V, int R, int k,
                                     const int32_t* draft_tokens, const int32_t* kv_lens_in,
                                     int32_t* argmax_ids, int32_t* accepted, int32_t* next_tokens,
                                     int32_t* kv_lens_out, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H_ */
